"""Slot spill to host memory and restore (needs a GB300).

Tempo9 docs, "KV cache spills to disk, by default": a reusable prefix leaves
device memory and comes back later; a record from another model or KV layout
is recognised by its configuration hash and refused.  Here the record lives
in pinned host memory.  The round trip is bit-exact, and a suffix prefilled
after a restore (into the same context or a fresh one) is bit-identical to
one prefilled without the round trip and matches the oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import oracle_dims, oracle_weights
from oracle import model as om

pytestmark = pytest.mark.gpu
TAG = 0x5eed


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def ctx(shape, cap, n_slots=2, max_rows=160, n_layers=None):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    return Kvr(config_for_shape(shape, n_slots, cap, max_rows, n_layers=n_layers), device="cuda")


def kv_snapshot(kv, slot, n):
    out = []
    for l in range(kv.cfg.n_layers):
        k, v = kv.kvr_slot_kv(slot, l)
        out.append((k[:, :n].clone(), v[:, :, :n].clone()))
    return out


@pytest.mark.parametrize("shape_name,P", [("small", 77), ("small_d128", 130)])
def test_spill_restore_round_trip_is_exact(shape_name, P):
    shape = workloads.SHAPES[shape_name]
    lws = workloads.stack_weights(shape, 21)
    gw = workloads.weights_to(lws, "cuda")
    toks = list(range(600, 600 + P + 20))
    x = workloads.hidden_for_tokens(toks, shape.hidden, 5)

    kv = ctx(shape, 256)
    w = kv.weights(gw)
    assert kv.kvr_slot_match(toks[:P]) == (0, 0)
    kv.kvr_prefill_suffix(0, toks[:P], x[:P].cuda(), w)
    before = kv_snapshot(kv, 0, P)
    rec = kv.kvr_slot_spill(0, TAG)
    hd = rec[:64].numpy()
    assert bytes(hd[:8]) == b"KVRSLOT1"
    L, Hkv, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    tok_bytes = -(-P * 4 // 16) * 16
    assert rec.numel() == 64 + tok_bytes + L * 2 * Hkv * P * d * 2
    assert rec[64:64 + 4 * P].view(torch.int32).tolist() == toks[:P]
    # layer 0's K section is the arena's K cut to P rows
    k0 = rec[64 + tok_bytes:64 + tok_bytes + Hkv * P * d * 2].view(torch.bfloat16).view(Hkv, P, d)
    assert torch.equal(k0, before[0][0].cpu())

    # the slot is reused for something else, then restored
    kv.kvr_slot_truncate(0, 0)
    other = list(range(9000, 9000 + P))
    kv.kvr_prefill_suffix(0, other, workloads.hidden_for_tokens(other, shape.hidden, 5).cuda(), w)
    kv.kvr_slot_restore(0, rec, TAG)
    assert kv.kvr_slot_len(0) == P and kv.kvr_slot_tokens(0) == toks[:P]
    for (k, v), (k0_, v0_) in zip(kv_snapshot(kv, 0, P), before):
        assert torch.equal(k, k0_) and torch.equal(v, v0_)
    # the match sees the restored prefix
    assert kv.kvr_slot_match(toks[:P + 20]) == (0, P)
    after = kv.kvr_prefill_suffix(0, toks[P:], x[P:].cuda(), w)

    # a context that never spilled gives the same bits; so does a fresh context
    # (another capacity and slot count) restored from the record
    ref = ctx(shape, 256)
    wr = ref.weights(gw)
    ref.kvr_slot_match(toks[:P])
    ref.kvr_prefill_suffix(0, toks[:P], x[:P].cuda(), wr)
    want = ref.kvr_prefill_suffix(0, toks[P:], x[P:].cuda(), wr)
    assert torch.equal(after, want)
    fresh = ctx(shape, 512, n_slots=3)
    wf = fresh.weights(gw)
    fresh.kvr_slot_restore(2, rec, TAG)
    got = fresh.kvr_prefill_suffix(2, toks[P:], x[P:].cuda(), wf)
    assert torch.equal(got, want)
    fresh.kvr_sync_status()

    # and the oracle agrees with the continued rows
    dims = oracle_dims(shape)
    W = [oracle_weights(shape, lw) for lw in lws]
    cache = om.SlotKV(L, Hkv, 256, d)
    whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    err = np.abs(workloads.bf16_to_f64(after) - whole[P:])
    assert (err <= 1e-2 + 2e-2 * np.abs(whole[P:])).all(), float(err.max())


def test_restore_refuses_other_models_and_damaged_records():
    from prefix_reused_prefill_gb300 import KvrError
    shape = workloads.SHAPES["small"]
    gw = workloads.weights_to(workloads.stack_weights(shape, 21), "cuda")
    kv = ctx(shape, 256)
    w = kv.weights(gw)
    toks = list(range(40, 140))
    kv.kvr_slot_match(toks)
    kv.kvr_prefill_suffix(0, toks, workloads.hidden_for_tokens(toks, shape.hidden, 5).cuda(), w)
    rec = kv.kvr_slot_spill(0, TAG)

    target = ctx(shape, 256)
    target.kvr_slot_assign(1, [1, 2, 3])

    def refused(code, record, tag=TAG, into=target):
        with pytest.raises(KvrError) as e:
            into.kvr_slot_restore(1, record, tag)
        assert e.value.code == code
        assert into.kvr_slot_tokens(1) == [1, 2, 3]   # unchanged

    refused(-7, rec, tag=TAG + 1)                       # other weights
    shallow = ctx(shape, 256, n_layers=1)               # other layout
    shallow.kvr_slot_assign(1, [1, 2, 3])
    refused(-7, rec, into=shallow)
    refused(-1, rec[:-16].clone())                      # truncated
    bad = rec.clone()
    bad[0] = ord("X")
    refused(-1, bad)                                    # not a record
    small_cap = ctx(shape, 64, max_rows=64)
    small_cap.kvr_slot_assign(1, [1, 2, 3])
    refused(-2, rec, into=small_cap)                    # 100 tokens > capacity 64
    # an empty slot spills to a header-only record and restores to length 0
    kv.kvr_slot_truncate(1, 0)
    empty = kv.kvr_slot_spill(1, TAG)
    assert empty.numel() == 64
    target.kvr_slot_restore(1, empty, TAG)
    assert target.kvr_slot_len(1) == 0
