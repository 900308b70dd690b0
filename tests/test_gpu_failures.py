"""Failure detection without a GPU fault (needs a GB300).

* Injected on the host (KVR_FAULT): an allocation failure refuses the
  context, a launch failure or a capacity failure refuses the call before
  anything is launched, and no slot changes.
* On the device: a wait that nothing completes gives up after its limit
  (1 s), the status word reports it, kvr_sync_status returns KVR_ERR_TIMEOUT
  and clears it, and the context keeps working (checked against the oracle).
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import oracle_dims, oracle_weights
from oracle import model as om

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def make(shape, fault=None, monkeypatch=None):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    if fault:
        monkeypatch.setenv("KVR_FAULT", fault)
    try:
        return Kvr(config_for_shape(shape, 2, 256, 64), device="cuda")
    finally:
        if fault:
            monkeypatch.delenv("KVR_FAULT")


def test_injected_allocation_failure_refuses_the_context(monkeypatch):
    from prefix_reused_prefill_gb300 import KvrError
    with pytest.raises(KvrError) as e:
        make(workloads.SHAPES["small"], "alloc", monkeypatch)
    assert e.value.code == -5


@pytest.mark.parametrize("fault,code", [("launch", -5), ("capacity", -2)])
def test_injected_call_failures_change_no_slot(monkeypatch, fault, code):
    from prefix_reused_prefill_gb300 import KvrError
    shape = workloads.SHAPES["small"]
    kv = make(shape, fault, monkeypatch)
    w = kv.weights(workloads.weights_to(workloads.stack_weights(shape, 21), "cuda"))
    kv.kvr_slot_assign(0, [1, 2, 3])
    x = workloads.hidden_for_tokens([4, 5], shape.hidden, 5).cuda()
    calls = [
        lambda: kv.kvr_prefill_suffix(0, [4, 5], x, w),
        lambda: kv.kvr_verify(0, [4, 5], x, w),
        lambda: kv.kvr_prefill_branches(0, [1, 1], [4, 5], x, w),
        lambda: kv.kvr_prefill_batch([0, 1], [[4], [5]], x, w),
    ]
    for call in calls:
        with pytest.raises(KvrError) as e:
            call()
        assert e.value.code == code
        assert kv.kvr_slot_tokens(0) == [1, 2, 3] and kv.kvr_slot_len(1) == 0


def test_device_wait_that_runs_out_is_reported_and_the_context_recovers():
    from prefix_reused_prefill_gb300 import KvrError
    shape = workloads.SHAPES["small"]
    lws = workloads.stack_weights(shape, 21)
    kv = make(shape)
    w = kv.weights(workloads.weights_to(lws, "cuda"))
    kv.kvr_sync_status()
    kv.kvr_selftest_wait()
    with pytest.raises(KvrError) as e:
        kv.kvr_sync_status()
    assert e.value.code == -4
    kv.kvr_sync_status()   # cleared
    # with the status word set, every later kernel of the call leaves at entry
    # (or at its next wait): a whole stack behind a wait that ran out costs
    # about one wait limit, not one per CTA and launch
    import time
    toks = list(range(300, 340))
    x = workloads.hidden_for_tokens(toks, shape.hidden, 5)
    t0 = time.time()
    kv.kvr_selftest_wait()
    kv.kvr_slot_match(toks)
    kv.kvr_prefill_suffix(0, toks, x.cuda(), w)   # 40 rows: GEMM, attention, epilogues
    kv.kvr_prefill_suffix(0, toks[:3], x[:3].cuda(), w)   # 3 rows: GEMV, split-KV
    with pytest.raises(KvrError) as e:
        kv.kvr_sync_status()
    assert e.value.code == -4
    assert time.time() - t0 < 5.0
    kv.kvr_sync_status()   # cleared
    # the context still computes the right thing (the skipped calls' rows are
    # cut away first)
    kv.kvr_slot_truncate(0, 0)
    s, reused = kv.kvr_slot_match(toks)
    assert reused == 0
    out = kv.kvr_prefill_suffix(s, toks, x.cuda(), w)
    kv.kvr_sync_status()
    dims = oracle_dims(shape)
    W = [oracle_weights(shape, lw) for lw in lws]
    cache = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    want = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), 0)
    err = np.abs(workloads.bf16_to_f64(out) - want)
    assert (err <= 1e-2 + 2e-2 * np.abs(want)).all()
