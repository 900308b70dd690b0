"""kvr_slot_match_static -- the match for callers with no device memory to lend.

Such callers (a router thread in a process whose device memory all belongs to
another component's caching allocator, or code that must not allocate while a
CUDA graph is being captured) cannot give the call a scratch area.  The entry
point stages its prompt copy and match lengths in a fixed array inside the
library instead.  This test drives it through the C ABI and checks that it
chooses exactly what kvr_slot_match chooses, on two calls in a row (the second
call finds the first call's leftovers in the array), and that prompts beyond
the array's limit are refused.  It sits in its own file so it runs last.
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _pair(n_slots, cap):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    cfg = config_for_shape(workloads.SHAPES["tiny"], n_slots, cap, 16)
    return Kvr(cfg, device="cuda"), Kvr(cfg, device="cuda")


def test_static_match_equals_match_on_two_calls_in_a_row():
    # turn-9 table: the first call cuts slot 0 back to 1668, the second call
    # (a shorter prompt from another conversation) must agree as well
    tk = workloads.turn9_tokens()
    a, b = _pair(4, 16384)
    for s in range(4):
        a.kvr_slot_assign(s, tk[f"slot{s}"])
        b.kvr_slot_assign(s, tk[f"slot{s}"])
    prompts = [tk["prompt"], tk["slot2"][:700] + list(range(50))]
    for p in prompts:
        want = a.kvr_slot_match(p)
        got = b.kvr_slot_match_static(p)
        assert got == want
        for s in range(4):
            assert b.kvr_slot_tokens(s) == a.kvr_slot_tokens(s)
    assert a.kvr_slot_match(tk["prompt"]) == b.kvr_slot_match_static(tk["prompt"])


def test_static_match_random_tables():
    rng = np.random.Generator(np.random.PCG64(4))
    for S in (1, 3, 4):
        a, b = _pair(S, 64)
        for trial in range(40):
            for s in range(S):
                if rng.random() < 0.7:
                    toks = rng.integers(0, 3, size=int(rng.integers(0, 64))).tolist()
                    a.kvr_slot_assign(s, toks)
                    b.kvr_slot_assign(s, toks)
            for _ in range(2):
                prompt = rng.integers(0, 3, size=int(rng.integers(1, 64))).tolist()
                assert b.kvr_slot_match_static(prompt) == a.kvr_slot_match(prompt)


def test_static_match_refuses_prompts_beyond_its_limit():
    from prefix_reused_prefill_gb300 import KvrError
    a, b = _pair(2, 16448)
    with pytest.raises(KvrError) as e:
        b.kvr_slot_match_static(list(range(16385)))
    assert e.value.code == -2 and "static match limit" in str(e.value)
    # at the limit, with a slot that matches the prompt up to its last token:
    # the kernel reads every word of the fixed prompt region
    # (slot 0 holds another conversation, so no empty slot takes the prompt)
    prompt = list(range(16384))
    held = prompt[:16383] + [99999]
    for kv in (a, b):
        kv.kvr_slot_assign(0, [7, 7, 7])
        kv.kvr_slot_assign(1, held)
    want = a.kvr_slot_match(prompt)
    assert want == (1, 16383)
    assert b.kvr_slot_match_static(prompt) == want
    assert b.kvr_slot_tokens(1) == a.kvr_slot_tokens(1) == prompt[:16383]
