"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in the oracle's source (a flipped sign, a
dropped term, a wrong index or operand, an off-by-one) on the CPU, runs every
pin of tests/test_oracle_{model,numerics,slots}.py against the mutant, and
requires at least one pin to fail.  A control run checks that the unmutated
oracle passes every pin through the same harness.
"""
import inspect
import textwrap

import numpy as np
import pytest

import test_oracle_model as pins_model
import test_oracle_numerics as pins_numerics
import test_oracle_slots as pins_slots
from oracle import formats, model, numerics, slots

PIN_MODULES = (pins_model, pins_numerics, pins_slots)


def _param_sets(f):
    sets = [{}]
    for mk in getattr(f, "pytestmark", []):
        if mk.name != "parametrize":
            continue
        names, values = mk.args[0], mk.args[1]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        new = []
        for base in sets:
            for v in values:
                vals = v if len(names) > 1 else (v,)
                new.append(dict(base, **dict(zip(names, vals))))
        sets = new
    return sets


def run_pins():
    """Names of the pins that fail (an exception of any kind counts)."""
    failed = []
    for mod in PIN_MODULES:
        for name in sorted(dir(mod)):
            if not name.startswith("test_"):
                continue
            f = getattr(mod, name)
            for kw in _param_sets(f):
                if "rng" in inspect.signature(f).parameters:
                    kw = dict(kw, rng=np.random.Generator(np.random.PCG64(1234)))
                try:
                    with np.errstate(all="ignore"):
                        f(**kw)
                except Exception:
                    failed.append(f"{mod.__name__}.{name}")
                    break
    return failed


def _mutant(owner, name, old, new):
    """owner.name (a module function or a class method) with `old` replaced by `new` in its source."""
    orig = getattr(owner, name)
    src = textwrap.dedent(inspect.getsource(orig))
    assert old == new or src.count(old) == 1, f"mutation anchor not unique in {name}: {old!r}"
    module = inspect.getmodule(orig)
    ns = dict(module.__dict__)
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    return orig, ns[name]


MUTATIONS = [
    # RoPE
    (model, "rope", "x1 * c - x2 * s", "x1 * c + x2 * s"),                    # rotation sign
    (model, "rope", "-2.0 * j / d", "-1.0 * j / d"),                           # frequency exponent
    (model, "rope", "x1, x2 = x[..., :half], x[..., half:]",
     "x1, x2 = x[..., 0::2], x[..., 1::2]"),                                     # interleaved pairs
    # attention
    (model, "attend", "keys @ q[h] / np.sqrt(d)", "keys @ q[h]"),               # dropped 1/sqrt(d)
    (model, "attend", "kv = h // group", "kv = h % K.shape[0]"),                # GQA head map
    (model, "attend", "o[h] = p @ V[kv, visible]", "o[h] = p @ K[kv, visible]"),  # K for V
    (model, "softmax", "e / np.sum(e)", "e / np.max(e)"),                       # normaliser
    # norm, FFN, residuals
    (model, "rmsnorm", "np.mean(h * h, axis=-1, keepdims=True)", "np.sum(h * h, axis=-1, keepdims=True)"),
    (model, "rmsnorm", "h / np.sqrt(ms + eps) * g", "h / np.sqrt(ms + eps)"),   # gain dropped
    (model, "layer", 'silu(linear(b, W["wg"])) * linear(b, W["wu"])',
     'silu(linear(b, W["wu"])) * linear(b, W["wg"])'),                          # gate <-> up
    (model, "layer", 'h = h + linear(o, W["wo"])', 'h = linear(o, W["wo"])'),  # attention residual
    (model, "layer", 'return h + linear(z, W["wd"])', 'return linear(z, W["wd"])'),  # FFN residual
    (model, "linear", "x @ w.T", "x @ w"),                                      # transposed operand
    # rows and positions
    (model, "plain_rows", "np.arange(p0 + i + 1)", "np.arange(p0 + i)"),       # row misses itself
    (model, "branch_rows", "Row(P + i, P + off + i, vis)", "Row(P + off + i, P + off + i, vis)"),
    (model, "branch_rows", "np.concatenate([np.arange(P), P + off + np.arange(i + 1)])",
     "np.concatenate([np.arange(P + off), P + off + np.arange(i + 1)])"),      # sees earlier branches
    # output head and greedy acceptance
    (model, "head_logits", "rmsnorm(np.asarray(h, dtype=np.float64), gain, dims.rms_eps)",
     "np.asarray(h, dtype=np.float64)"),                                         # final norm dropped
    (model, "greedy_argmax", "np.argmax(logits, axis=-1)",
     "logits.shape[-1] - 1 - np.argmax(logits[..., ::-1], axis=-1)"),           # ties to the highest index
    (model, "greedy_accept", "int(tokens[a + 1]) == int(argmax[a])", "int(tokens[a]) == int(argmax[a])"),
    (model, "greedy_accept", "while a + 1 < len(tokens)", "while a + 2 < len(tokens)"),  # last draft never taken
    # scalar numerics and formats
    (numerics, "round_bf16", "np.rint(", "np.trunc("),                          # truncation
    (numerics, "silu", "1.0 + np.exp(-x)", "1.0 + np.exp(x)"),
    (formats, "int4_codes", ".astype(np.int64) - 8", ".astype(np.int64)"),     # missing offset
    (formats, "int4_codes", "field = kk // 8 + 4 * (kk % 2)", "field = kk % 8"),  # nibble order
    (formats, "q4k_record_fields", "(x >> (6 * f)) & 63", "(x >> (6 * f)) & 31"),  # field width
    (formats, "q4k_record_fields", "fields[..., :8], fields[..., 8:]", "fields[..., 8:], fields[..., :8]"),
    (formats, "q4k_record_fields", "d = rec[..., 0:2]", "d = rec[..., 2:4]"),  # d from dmin's bytes
    (formats, "dequant_q4k", "- (dmin[:, :, None, None]", "+ (dmin[:, :, None, None]"),  # min sign
    (formats, "dequant_q4k", "int4_codes(packed, K) + 8", "int4_codes(packed, K)"),  # signed codes
    # slot policy
    (slots.SlotTable, "choose", "ok = l[best] > self.lcp_with_others(best)",
     "ok = l[best] >= self.lcp_with_others(best)"),                            # threshold
    (slots.SlotTable, "choose", "return best, min(l[best], n - 1), l", "return best, min(l[best], n), l"),
    (slots.SlotTable, "choose", "key=lambda s: self.stamp[s])", "key=lambda s: -self.stamp[s])"),  # MRU
    (slots.SlotTable, "choose", "if ok and empty and l[best] < len(self.tokens[best]):", "if False:"),
]


def test_unmutated_oracle_passes_every_pin():
    assert run_pins() == []


def _install(monkeypatch, owner, name, orig, bad):
    monkeypatch.setattr(owner, name, bad)
    # pin modules that imported the name directly see the replacement too
    for mod in PIN_MODULES:
        if getattr(mod, name, None) is orig:
            monkeypatch.setattr(mod, name, bad)


@pytest.mark.parametrize("owner,name", sorted({(m[0], m[1]) for m in MUTATIONS}, key=lambda t: t[1]),
                         ids=lambda v: v if isinstance(v, str) else "")
def test_recompiled_unchanged_source_passes_every_pin(monkeypatch, owner, name):
    """The mutation mechanism itself (re-executing a function's source in its
    module's namespace) changes nothing: a mutant fails for its mistake."""
    orig, same = _mutant(owner, name, "", "")
    _install(monkeypatch, owner, name, orig, same)
    assert run_pins() == []


@pytest.mark.parametrize("owner,name,old,new", MUTATIONS,
                         ids=[f"{m[1]}:{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_fails_a_pin(monkeypatch, owner, name, old, new):
    orig, bad = _mutant(owner, name, old, new)
    _install(monkeypatch, owner, name, orig, bad)
    failed = run_pins()
    assert failed, f"no pin catches the mutation {old!r} -> {new!r} in {name}"
