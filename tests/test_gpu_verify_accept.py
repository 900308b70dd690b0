"""Greedy verification through the output head (kvr_verify_accept) against the
oracle, through the C ABI (needs a GB300).

The draft chain comes from the oracle: after the committed prefix, row j is fed
token toks[j]; the first `a` drafts are the oracle's argmax of the row before
them, the next one differs from it, the rest are arbitrary.  Logits are compared
by their decision: the GPU's argmax of every row must reach within LOGIT_TOL of
the oracle's largest logit (the stated bar |gpu - oracle| <= 1e-2 + 2e-2*|oracle|
taken at that logit, once for each side of the comparison), and the chain is
drawn only where the decisions that fix the acceptance count have a larger gap
than that, so the count and the kept tokens are exact.
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import oracle_dims, oracle_weights
from oracle import formats
from oracle import model as om

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def logit_tol(top):
    return 2 * (1e-2 + 2e-2 * abs(top))


def gap(lg):
    s = np.sort(lg)
    return s[-1] - s[-2]


def head_for(shape, vocab, seed):
    """bf16 gain drawn in [0.5, 1.5) (so a dropped or misplaced gain shows) and the int4 LM head."""
    hw = workloads.head_weights(shape, seed, "cpu", vocab=vocab)
    g = np.random.Generator(np.random.PCG64([seed, 77])).uniform(0.5, 1.5, shape.hidden)
    gain = torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16)
    lm = hw["lm"]
    dev = {"norm": gain.cuda(), "lm": workloads.Int4Matrix(lm.packed.cuda(), lm.scales.cuda(), None)}
    return dev, gain.to(torch.float64).numpy(), formats.dequant_int4(lm.packed.numpy(), lm.scales.numpy())


def make(shape_name, cap, max_rows, vocab, seed=21, n_slots=2):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES[shape_name]
    lws = workloads.stack_weights(shape, seed)
    kv = Kvr(config_for_shape(shape, n_slots, cap, max_rows, vocab=vocab), device="cuda")
    w = kv.weights(workloads.weights_to(lws, "cuda"))
    W = [oracle_weights(shape, lw) for lw in lws]
    return shape, kv, w, W


def oracle_chain(dims, W, cache, P, t0, m, a, gain, lm, xseed):
    """Rows one at a time from position P (the cache holds the prefix): the
    tokens fed, each row's logits.  toks[j+1] = argmax(row j) for j < a, then a
    different token."""
    vocab = lm.shape[0]
    toks, logits = [t0], []
    for j in range(m):
        x = workloads.bf16_to_f64(workloads.hidden_for_tokens([toks[j]], dims.hidden, xseed))
        h = om.forward(dims, W, cache, x, om.plain_rows(P + j, 1), rounded=False)
        lg = om.head_logits(dims, h, gain, lm)[0]
        logits.append(lg)
        if j + 1 < m:
            g = int(np.argmax(lg))
            toks.append(g if j < a else (g + 1 + 7 * j) % vocab)
    return toks, np.stack(logits)


def clear(toks, logits, a):
    """The oracle's decisions that fix the acceptance count hold at the tolerance:
    rows before the first rejection have a clear argmax, and the rejected
    draft sits clearly below that row's best."""
    for j in range(min(a, len(logits))):
        if gap(logits[j]) <= logit_tol(logits[j].max()):
            return False
    if a + 1 < len(toks):
        lg = logits[a]
        return lg[toks[a + 1]] < lg.max() - logit_tol(lg.max())
    return True


def check_rows(nxt, logits, what):
    for j, (g, lg) in enumerate(zip(nxt, logits)):
        assert 0 <= g < lg.shape[0], f"{what} row {j}: index {g}"
        top = lg.max()
        assert lg[g] >= top - logit_tol(top), (f"{what} row {j}: gpu argmax {g} logit {lg[g]:.5f}, "
                                               f"oracle best {int(lg.argmax())} logit {top:.5f}")
        if gap(lg) > logit_tol(top):
            assert g == int(lg.argmax()), f"{what} row {j}"


@pytest.mark.parametrize("vocab,P,m,a", [
    (1000, 37, 1, 0),       # a plain decode step: no drafts
    (1000, 37, 6, 0),       # first draft rejected
    (1000, 50, 6, 3),
    (1000, 50, 6, 5),       # every draft accepted
    (32000, 70, 9, 4),      # 250 head tiles: several per CTA
    (4100, 20, 40, 2),      # two 32-row GEMV passes, ragged last tile
])
def test_verify_accept_matches_oracle(vocab, P, m, a):
    shape, kv, w, W = make("small", 256, 128, vocab)
    dims = oracle_dims(shape)
    head, gain, lm = head_for(shape, vocab, 31)
    xseed = 5
    prefix = list(range(400, 400 + P))
    xp = workloads.hidden_for_tokens(prefix, shape.hidden, xseed)
    base = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    om.prefill(dims, W, base, workloads.bf16_to_f64(xp), 0)
    # a first token whose decisions are clear at the tolerance
    for t0 in range(900, 1100):
        cache = _copy_kv(base)
        toks, logits = oracle_chain(dims, W, cache, P, t0, m, a, gain, lm, xseed)
        if clear(toks, logits, a):
            break
    else:
        pytest.fail("no draft chain with clear decisions")

    assert kv.kvr_slot_match(prefix) == (0, 0)
    kv.kvr_prefill_suffix(0, prefix, xp.cuda(), w)
    out = torch.empty((m, shape.hidden), dtype=torch.bfloat16, device="cuda")
    x = workloads.hidden_for_tokens(toks, shape.hidden, xseed)
    nxt, acc = kv.kvr_verify_accept(0, toks, x.cuda(), w, head, out=out)
    check_rows(nxt, logits, f"vocab={vocab} m={m}")
    want = om.greedy_accept(toks, [int(lg.argmax()) for lg in logits])
    assert want == min(a, m - 1)
    assert acc == want
    assert kv.kvr_slot_len(0) == P + 1 + acc
    assert kv.kvr_slot_tokens(0) == prefix + toks[:1 + acc]
    # the rows' outputs are kvr_verify's
    cache = _copy_kv(base)
    rows = om.prefill(dims, W, cache, workloads.bf16_to_f64(x), P)
    err = np.abs(workloads.bf16_to_f64(out) - rows)
    assert (err <= 1e-2 + 2e-2 * np.abs(rows)).all(), float(err.max())


def _copy_kv(kv):
    c = om.SlotKV(*kv.K.shape)
    c.K[...] = kv.K
    c.V[...] = kv.V
    return c


def test_two_verify_steps_continue_from_the_kept_tokens():
    """The second verify starts from the first one's next token at P + 1 + accepted; the
    rejected rows' K/V (still in the arena past the slot's length) are overwritten."""
    vocab, P = 2000, 45
    shape, kv, w, W = make("small", 256, 128, vocab)
    dims = oracle_dims(shape)
    head, gain, lm = head_for(shape, vocab, 32)
    xseed = 6
    prefix = list(range(300, 300 + P))
    xp = workloads.hidden_for_tokens(prefix, shape.hidden, xseed)
    base = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
    om.prefill(dims, W, base, workloads.bf16_to_f64(xp), 0)
    for t0 in range(1200, 1400):
        c1 = _copy_kv(base)
        toks1, lg1 = oracle_chain(dims, W, c1, P, t0, 5, 2, gain, lm, xseed)
        # the kept rows (three), then the second verify from the next token, on a cache holding only them
        c2 = _copy_kv(base)
        om.forward(dims, W, c2, workloads.bf16_to_f64(workloads.hidden_for_tokens(toks1[:3], shape.hidden, xseed)),
                   om.plain_rows(P, 3), rounded=False)
        t1 = int(lg1[2].argmax())
        toks2, lg2 = oracle_chain(dims, W, c2, P + 3, t1, 4, 3, gain, lm, xseed)
        if clear(toks1, lg1, 2) and gap(lg1[2]) > logit_tol(lg1[2].max()) and clear(toks2, lg2, 3):
            break
    else:
        pytest.fail("no draft chain with clear decisions")
    kv.kvr_slot_match(prefix)
    kv.kvr_prefill_suffix(0, prefix, xp.cuda(), w)
    n1, a1 = kv.kvr_verify_accept(0, toks1, workloads.hidden_for_tokens(toks1, shape.hidden, xseed).cuda(), w, head)
    assert a1 == 2 and n1[2] == t1
    n2, a2 = kv.kvr_verify_accept(0, toks2, workloads.hidden_for_tokens(toks2, shape.hidden, xseed).cuda(), w, head)
    check_rows(n2, lg2, "second verify")
    assert a2 == 3
    assert kv.kvr_slot_tokens(0) == prefix + toks1[:3] + toks2


def test_verify_accept_refuses_bad_heads():
    from prefix_reused_prefill_gb300 import KvrError
    shape, kv, w, W = make("small", 256, 128, 1000)
    head, _, _ = head_for(shape, 1000, 31)
    kv.kvr_slot_match([1, 2, 3])
    kv.kvr_prefill_suffix(0, [1, 2, 3], workloads.hidden_for_tokens([1, 2, 3], shape.hidden, 5).cuda(), w)
    x = workloads.hidden_for_tokens([4, 5], shape.hidden, 5).cuda()
    big, _, _ = head_for(shape, 1024, 31)   # more rows than the configured vocab
    with pytest.raises(KvrError):
        kv.kvr_verify_accept(0, [4, 5], x, w, big)
    assert kv.kvr_slot_len(0) == 3
    with pytest.raises(KvrError):
        kv.kvr_verify_accept(0, list(range(65)), torch.zeros(65, shape.hidden, dtype=torch.bfloat16).cuda(),
                             w, head)
    assert kv.kvr_slot_len(0) == 3
    nxt, acc = kv.kvr_verify_accept(0, [4, 5], x, w, head)
    assert kv.kvr_slot_len(0) == 3 + 1 + acc and len(nxt) == 2


def test_batched_verify_accept_matches_each_conversation():
    """Three conversations in one kvr_verify_accept_batch call: every row's
    decision, each acceptance count and each slot's kept tokens as the oracle
    gives them for the conversation alone."""
    vocab = 1000
    shape, kv, w, W = make("small", 256, 128, vocab, n_slots=3)
    dims = oracle_dims(shape)
    head, gain, lm = head_for(shape, vocab, 33)
    xseed = 7
    plan = [(2, 41, 5, 2), (0, 60, 1, 0), (1, 23, 4, 3)]   # (slot, P, m, a)
    toks_all, logits_all, prefixes = [], [], []
    for slot, P, m, a in plan:
        prefix = list(range(100 * (slot + 1), 100 * (slot + 1) + P))
        xp = workloads.hidden_for_tokens(prefix, shape.hidden, xseed)
        base = om.SlotKV(shape.n_layers, shape.n_kv_heads, 256, shape.head_dim)
        om.prefill(dims, W, base, workloads.bf16_to_f64(xp), 0)
        for t0 in range(700 + 50 * slot, 900 + 50 * slot):
            toks, logits = oracle_chain(dims, W, _copy_kv(base), P, t0, m, a, gain, lm, xseed)
            if clear(toks, logits, a):
                break
        else:
            pytest.fail("no draft chain with clear decisions")
        kv.kvr_prefill_suffix(slot, prefix, xp.cuda(), w)
        toks_all.append(toks)
        logits_all.append(logits)
        prefixes.append(prefix)
    x = torch.cat([workloads.hidden_for_tokens(t, shape.hidden, xseed) for t in toks_all]).contiguous()
    nxt, acc = kv.kvr_verify_accept_batch([p[0] for p in plan], toks_all, x.cuda(), w, head)
    for (slot, P, m, a), toks, logits, prefix, n, got in zip(plan, toks_all, logits_all, prefixes, nxt, acc):
        check_rows(n, logits, f"batched slot {slot}")
        assert got == min(a, m - 1)
        assert kv.kvr_slot_tokens(slot) == prefix + toks[:1 + got]
