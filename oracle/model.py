"""The decoder stack of the suffix prefill, evaluated plainly in float64.

TEST INFRASTRUCTURE ONLY (see the package header).

Sources: goinfer, "Turn nine in under half a second" ("What goinfer does": each
conversation keeps one key and one value row per token and layer, and a prompt
runs only past the part the conversation already holds; "What we got wrong": a
speculative step checks the guessed tokens and must give the same words as
plain decoding); the spec-decode post ("cost model": the m = k+1 verify rows
run as one batched pass over weights read once); OpenJev "What changed" (several questions resume from one shared
checkpoint).  The pages do not print the layer; the layer below is the
pre-norm Qwen2-style decoder those pages serve (RMSNorm, GQA attention with
rotate-half RoPE, SwiGLU), with the readings listed in the design notes:

* rows are at absolute slot positions: a cached row and a recomputed row of
  the same token at the same position are the same row;
* bf16 rounding happens where the model stores a bf16 tensor: the normed
  activations a and b, q/k/v after RoPE, the attention output, the SwiGLU
  product, the final output.  Everything else is float64.  The residual
  stream is not rounded inside one call.
* query head h reads KV head h // (Hq/Hkv);
* the scores are q.k / sqrt(d), softmax with the row maximum subtracted.

Parity pins (tests/test_oracle_model.py): constant V per KV head gives that
constant; q = 0 gives the plain mean of the visible V rows; one row at
position 0 gives v_0; softmax rows sum to 1; RoPE preserves norms, is the
identity at position 0, makes q.k depend only on the position difference, and
matches a worked example (tests/golden/rope_fixture.txt); RMSNorm is
invariant to positive scaling and maps a constant vector to ~1; a layer whose
Wo and Wd are zero is the identity; prefill(whole) == prefill(prefix) then
prefill(suffix), bit for bit; the branch rows of a priming batch equal
separate truncate-and-prefill runs, bit for bit; layer_rows equals layer on
the rows it evaluates, bit for bit; greedy acceptance on hand-worked token
lists; the head with an identity LM head ranks the normed stream, and a
one-row head is that row's dot product.  The stack as a whole beyond
these invariants is "parity unpinned": no page prints a worked numeric
example of a layer.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Sequence

import numpy as np

from .numerics import round_bf16, silu


@dataclasses.dataclass(frozen=True)
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    attn_only: bool
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


class SlotKV:
    """K and V of one slot for every layer: float64 [L][Hkv][cap][d], bf16-valued."""

    def __init__(self, n_layers: int, n_kv_heads: int, cap: int, head_dim: int):
        self.K = np.zeros((n_layers, n_kv_heads, cap, head_dim))
        self.V = np.zeros((n_layers, n_kv_heads, cap, head_dim))


@dataclasses.dataclass
class Row:
    pos: int            # RoPE position
    store: int          # index in the slot where its K/V are written
    visible: np.ndarray  # slot indices of the keys this row attends to


def plain_rows(p0: int, m: int) -> List[Row]:
    """Suffix / verify rows: row i sits at p0+i and sees keys 0..p0+i."""
    return [Row(p0 + i, p0 + i, np.arange(p0 + i + 1)) for i in range(m)]


def branch_rows(P: int, lens: Sequence[int]) -> List[Row]:
    """Priming rows: branch b's row i sits at position P+i (as if it were the
    only question), is stored after every earlier branch's rows, and sees the
    shared state [0, P) plus its own branch's rows up to itself."""
    rows, off = [], 0
    for n in lens:
        for i in range(n):
            vis = np.concatenate([np.arange(P), P + off + np.arange(i + 1)])
            rows.append(Row(P + i, P + off + i, vis))
        off += n
    return rows


# ----------------------------------------------------------------------------
# pieces of a layer
# ----------------------------------------------------------------------------

def rmsnorm(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) * g over the last axis."""
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [heads][d] at one position.

    Pair (j, j + d/2) is rotated by the angle pos * theta**(-2j/d).
    """
    d = x.shape[-1]
    half = d // 2
    j = np.arange(half, dtype=np.float64)
    ang = pos * np.power(theta, -2.0 * j / d)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s: np.ndarray) -> np.ndarray:
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray, group: int) -> np.ndarray:
    """One row: q [Hq][d]; K, V [Hkv][cap][d] of one layer -> o [Hq][d]."""
    Hq, d = q.shape
    o = np.empty_like(q)
    for h in range(Hq):
        kv = h // group
        keys = K[kv, visible]                 # [n][d]
        p = softmax(keys @ q[h] / np.sqrt(d))
        o[h] = p @ V[kv, visible]
    return o


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x [m][K] times w [N][K] transposed -> [m][N]."""
    return x @ w.T


def layer(dims: Dims, W: Dict[str, np.ndarray], h: np.ndarray, K: np.ndarray, V: np.ndarray,
          rows: List[Row]) -> np.ndarray:
    """One decoder layer over the rows; writes their K/V into K, V (one layer).

    h is the layer input [m][H] (float64).  Returns the layer output.
    """
    Hq, Hkv, d = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    if dims.attn_only:
        a = h
    else:
        a = round_bf16(rmsnorm(h, W["norm_attn"], dims.rms_eps))
    q = linear(a, W["wq"]).reshape(-1, Hq, d)
    k = linear(a, W["wk"]).reshape(-1, Hkv, d)
    v = linear(a, W["wv"]).reshape(-1, Hkv, d)
    qs = []
    for i, r in enumerate(rows):
        qs.append(round_bf16(rope(q[i], r.pos, dims.rope_theta)))
        K[:, r.store] = round_bf16(rope(k[i], r.pos, dims.rope_theta))
        V[:, r.store] = round_bf16(v[i])
    o = np.stack([round_bf16(attend(qs[i], K, V, r.visible, dims.group)).reshape(Hq * d)
                  for i, r in enumerate(rows)])
    if dims.attn_only:
        return round_bf16(linear(o, W["wo"]))
    h = h + linear(o, W["wo"])
    b = round_bf16(rmsnorm(h, W["norm_ffn"], dims.rms_eps))
    z = round_bf16(silu(linear(b, W["wg"])) * linear(b, W["wu"]))
    return h + linear(z, W["wd"])


def layer_rows(dims: Dims, W: Dict[str, np.ndarray], h: np.ndarray, K: np.ndarray, V: np.ndarray,
               rows: List[Row], out_rows: Sequence[int]) -> np.ndarray:
    """The same layer, evaluated only for the rows listed in out_rows.

    A row's output depends on the other rows only through their K/V, so K/V
    are computed (and written into K, V) for every row, and the query,
    attention, O projection and FFN only for out_rows.  Returns
    [len(out_rows)][H].  Bit-identical to ``layer`` on those rows (pinned).
    """
    Hq, Hkv, d = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    if dims.attn_only:
        a = h
    else:
        a = round_bf16(rmsnorm(h, W["norm_attn"], dims.rms_eps))
    k = linear(a, W["wk"]).reshape(-1, Hkv, d)
    v = linear(a, W["wv"]).reshape(-1, Hkv, d)
    for i, r in enumerate(rows):
        K[:, r.store] = round_bf16(rope(k[i], r.pos, dims.rope_theta))
        V[:, r.store] = round_bf16(v[i])
    sel = list(out_rows)
    q = linear(a[sel], W["wq"]).reshape(-1, Hq, d)
    o = np.stack([round_bf16(attend(round_bf16(rope(q[n], rows[i].pos, dims.rope_theta)), K, V,
                                    rows[i].visible, dims.group)).reshape(Hq * d)
                  for n, i in enumerate(sel)])
    if dims.attn_only:
        return round_bf16(linear(o, W["wo"]))
    hs = h[sel] + linear(o, W["wo"])
    b = round_bf16(rmsnorm(hs, W["norm_ffn"], dims.rms_eps))
    z = round_bf16(silu(linear(b, W["wg"])) * linear(b, W["wu"]))
    return hs + linear(z, W["wd"])


def forward(dims: Dims, weights: List[Dict[str, np.ndarray]], kv: SlotKV, hidden: np.ndarray,
            rows: List[Row], rounded: bool = True) -> np.ndarray:
    """Run the rows through every layer; K/V land in ``kv``.  Returns the
    bf16-valued output [m][H] (the final residual stream, rounded once), or
    the unrounded stream with rounded=False."""
    h = np.asarray(hidden, dtype=np.float64)
    for l, W in enumerate(weights):
        h = layer(dims, W, h, kv.K[l], kv.V[l], rows)
    return round_bf16(h) if rounded else h


# ----------------------------------------------------------------------------
# the output head and greedy verification
# ----------------------------------------------------------------------------

def head_logits(dims: Dims, h: np.ndarray, gain: np.ndarray, w_lm: np.ndarray) -> np.ndarray:
    """Logits [m][vocab] of output rows: the final RMSNorm (rounded to bf16, as
    every normed activation) times the LM head."""
    b = round_bf16(rmsnorm(np.asarray(h, dtype=np.float64), gain, dims.rms_eps))
    return linear(b, w_lm)


def greedy_argmax(logits: np.ndarray) -> np.ndarray:
    """Index of each row's largest logit; ties go to the lowest index."""
    return np.argmax(logits, axis=-1)


def greedy_accept(tokens: Sequence[int], argmax: Sequence[int]) -> int:
    """Verify rows hold [t0, d1 .. dk]: draft d_(j+1) is accepted while it
    equals the argmax of row j (greedy decoding would have produced it).
    Returns the number of accepted drafts; the next token is argmax[accepted]."""
    a = 0
    while a + 1 < len(tokens) and int(tokens[a + 1]) == int(argmax[a]):
        a += 1
    return a


def verify_accept(dims: Dims, weights, kv: SlotKV, hidden: np.ndarray, p0: int, tokens: Sequence[int],
                  gain: np.ndarray, w_lm: np.ndarray):
    """Verify the m rows at p0 .. p0+m-1 and take the greedy decision.
    Returns (logits, argmax, accepted)."""
    h = forward(dims, weights, kv, hidden, plain_rows(p0, len(hidden)), rounded=False)
    logits = head_logits(dims, h, gain, w_lm)
    am = greedy_argmax(logits)
    return logits, am, greedy_accept(tokens, am)


def prefill(dims: Dims, weights, kv: SlotKV, hidden: np.ndarray, p0: int) -> np.ndarray:
    """Suffix prefill (and speculative verify): m rows at p0 .. p0+m-1."""
    return forward(dims, weights, kv, hidden, plain_rows(p0, len(hidden)))


def prefill_branches(dims: Dims, weights, kv: SlotKV, hidden: np.ndarray, P: int,
                     lens: Sequence[int]) -> np.ndarray:
    """Several questions resuming from the checkpoint at P, in one batch."""
    assert sum(lens) == len(hidden)
    return forward(dims, weights, kv, hidden, branch_rows(P, lens))
