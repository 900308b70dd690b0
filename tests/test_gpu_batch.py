"""Several conversations in one call (kvr_prefill_batch) against the oracle
(needs a GB300).

Each conversation appends its rows to its own slot after that slot's cached
tokens; the oracle runs each conversation alone on its own cache.  Outputs and
the K/V written to every slot are compared elementwise at the stated bar
|gpu - oracle| <= 1e-2 + 2e-2*|oracle|; lengths and token lists are exact.
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
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} out of tolerance, max err {err.max():.4g}"


@pytest.mark.parametrize("shape_name,prefixes,lens", [
    ("small", [37, 90, 0, 64], [1, 5, 3, 8]),          # 17 rows: GEMV, split-KV attention
    ("small", [20, 0, 130, 45], [30, 1, 40, 7]),       # 78 rows: tcgen05 GEMM; 30 and 40 rows take tcgen05 attention
    ("small_d128", [50, 11], [4, 2]),
    ("small_bf16", [33, 70, 5], [2, 9, 1]),
    ("small_q4k", [40, 9], [3, 50]),
])
def test_batch_matches_each_conversation_alone(shape_name, prefixes, lens):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES[shape_name]
    n = len(lens)
    lws = workloads.stack_weights(shape, 21)
    kv = Kvr(config_for_shape(shape, 4, 256, 160), device="cuda")
    w = kv.weights(workloads.weights_to(lws, "cuda"))
    dims = oracle_dims(shape)
    W = [oracle_weights(shape, lw) for lw in lws]
    # conversation j lives in slot order[j] (not in slot order)
    order = [3, 1, 0, 2][:n]
    seqs = [list(range(1000 * (j + 1), 1000 * (j + 1) + prefixes[j] + lens[j])) for j in range(n)]
    xs = [workloads.hidden_for_tokens(s, shape.hidden, 5 + j) for j, s in enumerate(seqs)]
    for j in range(n):
        if prefixes[j]:
            kv.kvr_prefill_suffix(order[j], seqs[j][:prefixes[j]], xs[j][:prefixes[j]].cuda(), w)
    rows = [s[p:] for s, p in zip(seqs, prefixes)]
    hid = torch.cat([x[p:] for x, p in zip(xs, prefixes)]).contiguous()
    out = kv.kvr_prefill_batch(order, rows, hid.cuda(), w)
    kv.kvr_sync_status()
    at = 0
    for j in range(n):
        s, P, m = order[j], prefixes[j], lens[j]
        assert kv.kvr_slot_len(s) == P + m and kv.kvr_slot_tokens(s) == seqs[j]
        cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
        whole = om.prefill(dims, W, cache, workloads.bf16_to_f64(xs[j]), 0)
        close(workloads.bf16_to_f64(out[at:at + m]), whole[P:], f"conversation {j} rows")
        for l in range(shape.n_layers):
            k, v = kv.kvr_slot_kv(s, l)
            close(workloads.bf16_to_f64(k[:, :P + m]), cache.K[l][:, :P + m], f"conversation {j} K layer {l}")
            close(workloads.bf16_to_f64(v[:, :, :P + m].transpose(1, 2)), cache.V[l][:, :P + m],
                  f"conversation {j} V layer {l}")
        at += m


def test_batch_refuses_bad_requests_and_changes_nothing():
    from prefix_reused_prefill_gb300 import Kvr, KvrError, config_for_shape
    shape = workloads.SHAPES["small"]
    kv = Kvr(config_for_shape(shape, 3, 128, 64), device="cuda")
    w = kv.weights(workloads.weights_to(workloads.stack_weights(shape, 21), "cuda"))
    for a in (0, 50):   # 100 cached tokens in slot 0 (max_rows 64 per call)
        t = list(range(a, a + 50))
        kv.kvr_prefill_suffix(0, t, workloads.hidden_for_tokens(t, shape.hidden, 5).cuda(), w)
    x = lambda n: torch.zeros(n, shape.hidden, dtype=torch.bfloat16).cuda()
    cases = [
        ([1, 1], [[5], [6]], -1),                 # a slot twice
        ([0, 1], [list(range(29)), [7]], -2),     # 100 + 29 > capacity 128
        ([1, 2], [list(range(40)), list(range(30))], -2),   # 70 rows > max_rows 64
        ([1, 5], [[5], [6]], -1),                 # no such slot
    ]
    for slots, toks, code in cases:
        with pytest.raises(KvrError) as e:
            kv.kvr_prefill_batch(slots, toks, x(sum(len(t) for t in toks)), w)
        assert e.value.code == code
        assert [kv.kvr_slot_len(s) for s in range(3)] == [100, 0, 0]
