"""The persistent small-m pass against the oracle and against the per-step launches.

With KVR_PASS=1, calls with up to 16 rows of an int4 stack with head_dim 128
run as one cooperative launch (k_pass.cu); by default (KVR_PASS unset or 0)
they stay on the per-step GEMV and attention launches.  Both are checked against the oracle with the stated
elementwise bound, and against each other, over a prefix of several 64-key
blocks (several key splits per KV head), for row counts across the one- and
two-n-tile variants, branch rows, consecutive calls with changing row counts,
and the greedy output head.
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import oracle_dims, oracle_weights
from oracle import model as om

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} out of tolerance, max err {err.max():.4g}"
    return float(err.max())


def make(monkeypatch, use_pass, shape_name="small_g4", cap=1024, max_rows=256, n_slots=2, seed=21):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    monkeypatch.setenv("KVR_PASS", "1" if use_pass else "0")
    shape = workloads.SHAPES[shape_name]
    lws = workloads.stack_weights(shape, seed)
    kv = Kvr(config_for_shape(shape, n_slots, cap, max_rows, vocab=workloads.VOCAB), device="cuda")
    monkeypatch.delenv("KVR_PASS")
    w = kv.weights(workloads.weights_to(lws, "cuda"))
    return shape, kv, w, [oracle_weights(shape, lw) for lw in lws], lws


def slot_kv(kv, slot, layer, n):
    k, v = kv.kvr_slot_kv(slot, layer)
    return workloads.bf16_to_f64(k[:, :n]), workloads.bf16_to_f64(v[:, :, :n].transpose(1, 2))


@pytest.mark.parametrize("P", [0, 77, 700])
def test_pass_matches_oracle_and_the_per_step_launches(monkeypatch, P):
    toks = list(range(500, 500 + P + 16))
    outs = {}
    for use_pass in (True, False):
        shape, kv, w, W, _ = make(monkeypatch, use_pass)
        x = workloads.hidden_for_tokens(toks, shape.hidden, 5)
        dims = oracle_dims(shape)
        cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 1024, shape.head_dim)
        whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
        kv.kvr_slot_match(toks[:1] if P else [toks[0]])
        for a in range(0, P, 256):
            b = min(P, a + 256)
            kv.kvr_prefill_suffix(0, toks[a:b], x[a:b].cuda(), w)
        for m in (1, 2, 4, 7, 8, 9, 16):
            kv.kvr_slot_truncate(0, P)
            out = kv.kvr_prefill_suffix(0, toks[P:P + m], x[P:P + m].cuda(), w)
            kv.kvr_sync_status()
            got = workloads.bf16_to_f64(out)
            close(got, whole[P:P + m], f"pass={use_pass} P={P} m={m}")
            outs[(use_pass, m)] = got
            for l in range(shape.n_layers):
                k, v = slot_kv(kv, 0, l, P + m)
                close(k[:, P:], cache.K[l][:, P:P + m], f"pass={use_pass} P={P} m={m} K layer {l}")
                close(v[:, P:], cache.V[l][:, P:P + m], f"pass={use_pass} P={P} m={m} V layer {l}")
        kv.close()
    for m in (1, 2, 4, 7, 8, 9, 16):
        close(outs[(True, m)], outs[(False, m)], f"pass vs per-step launches P={P} m={m}")


def test_pass_branches_and_consecutive_calls(monkeypatch):
    shape, kv, w, W, _ = make(monkeypatch, True)
    dims = oracle_dims(shape)
    P = 130
    state = list(range(7, 7 + P))
    qs = [[3000 + i for i in range(3)], [4000 + i for i in range(5)]]
    xs = workloads.hidden_for_tokens(state, shape.hidden, 5)
    xq = workloads.hidden_for_tokens(sum(qs, []), shape.hidden, 5)
    kv.kvr_slot_match(state)
    kv.kvr_prefill_suffix(0, state, xs.cuda(), w)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 1024, shape.head_dim)
    om.prefill(dims, W, cache, workloads.bf16_to_f64(xs), 0)
    ref = om.prefill_branches(dims, W, cache, workloads.bf16_to_f64(xq), P, [3, 5])
    for rep in range(3):   # the same call again: completion counters of earlier calls stay behind
        out = kv.kvr_prefill_branches(0, [3, 5], sum(qs, []), xq.cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), ref, f"branches, call {rep}")
        assert kv.kvr_slot_len(0) == P
    # then one-row steps that commit, each continuing from the last
    toks = state + list(range(9000, 9006))
    x = workloads.hidden_for_tokens(toks, shape.hidden, 5)
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 1024, shape.head_dim)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    for i in range(P, P + 6):
        out = kv.kvr_prefill_suffix(0, toks[i:i + 1], x[i:i + 1].cuda(), w)
        kv.kvr_sync_status()
        close(workloads.bf16_to_f64(out), whole[i:i + 1], f"one-row step at {i}")
    kv.close()


def test_pass_with_the_greedy_head(monkeypatch):
    """kvr_verify_accept through the pass: the final norm is formed in the pass,
    the LM head and the decision follow; decisions equal those of the per-step
    launches."""
    res = {}
    for use_pass in (True, False):
        shape, kv, w, W, lws = make(monkeypatch, use_pass)
        vocab = 4096
        hw = workloads.head_weights(shape, 21, "cpu", vocab=vocab)
        head = {"norm": hw["norm"].cuda(),
                "lm": workloads.Int4Matrix(hw["lm"].packed.cuda(), hw["lm"].scales.cuda(), None)}
        toks = list(range(200, 200 + 90))
        x = workloads.hidden_for_tokens(toks, shape.hidden, 5)
        kv.kvr_slot_match(toks[:1])
        kv.kvr_prefill_suffix(0, toks[:80], x[:80].cuda(), w)
        got = []
        for m in (1, 5, 10):
            nxt, acc = kv.kvr_verify_accept(0, toks[80:80 + m], x[80:80 + m].cuda(), w, head)
            got.append((list(nxt), acc, kv.kvr_slot_len(0)))
            kv.kvr_slot_truncate(0, 80)
        res[use_pass] = got
        kv.close()
    assert res[True] == res[False]
