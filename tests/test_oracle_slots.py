"""Pins of the oracle's slot policy (no GPU)."""
import itertools

import numpy as np
import pytest

import workloads
from oracle.slots import SlotTable, common_prefix


def brute_choice(slots, stamps, prompt, threshold=True):
    """Brute-force reading of goinfer's rule on a tiny table.

    A slot "holds the start of the prompt" for the longest L with
    slot[:L] == prompt[:L]; a candidate must share more with the prompt than
    with any other occupied slot, and may not cut its slot back while another
    slot is empty; the longest candidate wins; otherwise the first empty
    slot, and with none empty the slot whose last use is oldest.
    """
    def shared(a, b):
        return max(L for L in range(min(len(a), len(b)) + 1) if list(a[:L]) == list(b[:L]))

    occ = [s for s in range(len(slots)) if slots[s] is not None]
    any_empty = len(occ) < len(slots)
    cands = []
    for s in occ:
        l = shared(slots[s], prompt)
        o = max([shared(slots[s], slots[t]) for t in occ if t != s] + [0])
        if l > 0 and (not threshold or (l > o and not (any_empty and l < len(slots[s])))):
            cands.append((l, s))
    if threshold and cands:
        best = max(c[0] for c in cands)
        assert sum(1 for c in cands if c[0] == best) == 1, "R1: an accepted best slot is unique"
    if cands:
        # the best slot overall must itself be a candidate (R1's first consequence)
        l_all = {s: shared(slots[s], prompt) for s in occ}
        lmax = max(l_all.values())
        l, s = max(cands, key=lambda c: (c[0], -c[1]))
        if threshold:
            assert l == lmax
        return s, min(l, len(prompt) - 1)
    empties = [s for s in range(len(slots)) if slots[s] is None]
    if empties:
        return empties[0], 0
    return min(range(len(slots)), key=lambda s: stamps[s]), 0


@pytest.mark.parametrize("threshold", [True, False])
def test_policy_matches_brute_force(threshold):
    rng = np.random.Generator(np.random.PCG64(77))
    for trial in range(3000):
        S = int(rng.integers(1, 5))
        vocab = int(rng.integers(2, 5))
        t = SlotTable(S, 12, threshold)
        for s in range(S):
            if rng.random() < 0.8:
                t.assign(s, rng.integers(0, vocab, size=int(rng.integers(0, 12))).tolist())
        # scramble LRU stamps
        for s in rng.permutation(S):
            if t.tokens[s] is not None:
                t._touch(int(s))
        prompt = rng.integers(0, vocab, size=int(rng.integers(1, 12))).tolist()
        want = brute_choice(list(t.tokens), list(t.stamp), prompt, threshold)
        got = t.choose(prompt)[:2]
        assert got == want, (trial, t.tokens, prompt)


def test_turn9_reuses_1668_tokens():
    tk = workloads.turn9_tokens()
    assert len(tk["prompt"]) == 1922
    t = SlotTable(4, 16384)
    for s in range(4):
        t.assign(s, tk[f"slot{s}"])
    slot, reused = t.match(tk["prompt"])
    assert (slot, reused) == (0, 1668)
    assert t.length(0) == 1668
    t.append(0, tk["prompt"][1668:])
    assert t.length(0) == 1922


def test_tiny_config_matches_slot0_at_90():
    tk = workloads.tiny_tokens()
    t = SlotTable(2, 256)
    t.assign(0, tk["slot0"]); t.assign(1, tk["slot1"])
    assert t.match(tk["prompt"]) == (0, 90)


def test_repeated_prompt_reuses_all_but_one():
    t = SlotTable(2, 64)
    t.serve_turn([5, 6, 7, 8])
    assert t.match([5, 6, 7, 8]) == (0, 3)
    # a cut-back while slot 1 is empty is a new conversation (R1b)
    assert t.choose([5, 6])[:2] == (1, 0)
    t.assign(1, [9, 9])
    assert t.match([5, 6]) == (0, 1)


def test_two_conversations_sharing_a_template_do_not_thrash():
    # "What we got wrong": two conversations taking turns, both starting with the
    # same 7-token template, must each keep their own slot and reuse their history
    rng = np.random.Generator(np.random.PCG64(5))
    tmpl = rng.integers(0, 1000, 7).tolist()
    conv = {c: tmpl + rng.integers(1000 * (c + 1), 1000 * (c + 2), 20).tolist() for c in (0, 1)}
    t = SlotTable(2, 4096)
    prev = {}
    for turn in range(6):
        for c in (0, 1):
            slot, prefilled = t.serve_turn(conv[c])
            reused = len(conv[c]) - prefilled
            if turn > 0:
                assert reused == prev[c]          # the whole previous history, not 7
                assert slot == c
            prev[c] = len(conv[c])
            conv[c] = conv[c] + rng.integers(1000 * (c + 1), 1000 * (c + 2), 13).tolist()
    # with the threshold off the first prompt after the other conversation steals its slot
    t = SlotTable(2, 4096, threshold=False)
    t.serve_turn(tmpl + [1, 2, 3])
    slot, _ = t.serve_turn(tmpl + [9, 9])
    assert slot == 0


def test_client_prefill_counts():
    # "What was measured": with enough slots each turn after the first prefills only
    # the new message; with one slot and several clients, the whole history again
    for clients, slots in [(1, 4), (2, 4), (4, 4), (4, 1)]:
        rng = np.random.Generator(np.random.PCG64(100 + clients))
        tmpl = rng.integers(0, 50, 7).tolist()
        convs = [tmpl + rng.integers(100, 32000, 30).tolist() for _ in range(clients)]
        t = SlotTable(slots, 16384)
        added = [len(c) for c in convs]
        for turn in range(6):
            for c in range(clients):
                slot, prefilled = t.serve_turn(convs[c])
                if turn > 0:
                    if slots >= clients:
                        assert prefilled == added[c]
                    elif clients > 1:
                        # one slot, several clients: the whole history beyond the template
                        assert prefilled == len(convs[c]) - len(tmpl)
                reply = rng.integers(100, 32000, 8).tolist()
                t.append(slot, reply)
                msg = rng.integers(100, 32000, int(rng.integers(12, 25))).tolist()
                convs[c] = convs[c] + reply + msg
                added[c] = len(msg)


def test_reuse_off_with_zero_slots():
    t = SlotTable(0, 64)
    t.serve_turn([1, 2, 3])
    assert t.match([1, 2, 3, 4]) == (0, 0)


def test_common_prefix():
    assert common_prefix([1, 2, 3], [1, 2, 4]) == 2
    assert common_prefix([], [1]) == 0
    assert common_prefix([1, 2], [1, 2, 3]) == 2
