"""Seeded synthetic inputs for the suffix-prefill workloads.

This module draws the random inputs that both the CUDA path and the oracle
consume: token lists for the slot table, per-token hidden states, and layer
weights.  It holds none of the method's arithmetic.  What it does do, because
an input has to be *in* the library's formats before anyone can read it:

* round N(0, 1) / N(0, 0.02) draws to bf16 (through torch's own cast);
* quantise N(0, 0.02) draws to the int4 group-32 format with fp16 scales and
  pack the 4-bit codes into the byte layout that ``include/kvr.h`` documents;
* draw the RMSNorm gains, bf16 in [0.5, 1.5), one set per norm.

The shapes are the ones the pages' workloads name (goinfer's turn-9 replay of
Qwen2.5-7B served as int4; the dense 9B of the speculative-decoding post; the
4B "balanced" profile of the prefix-priming page), with random weights because
no trained weights are in scope.

Randomness:
* small inputs come from numpy PCG64 (stable across machines);
* the per-token hidden state of token t is drawn from PCG64([seed, t]), so a
  token has the same hidden state in every call (the cached rows of a slot and
  the matching rows of a later prompt agree);
* full-size layer weights (gigabytes) are drawn on the requested device with a
  seeded torch generator; small test shapes draw them on the CPU.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

VOCAB = 32000
GROUP = 32  # int4 group size along the input (K) dimension


@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    n_layers: int
    weight_format: str  # "bf16" or "int4"
    attn_only: bool = False  # out = Attn(x) Wo^T, no norms / FFN / residual
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def matrices(self) -> Dict[str, tuple]:
        """(rows N, cols K) of every projection of one layer, torch Linear layout."""
        H, F = self.hidden, self.ffn
        m = {"wq": (self.q_dim, H), "wk": (self.kv_dim, H), "wv": (self.kv_dim, H),
             "wo": (H, self.q_dim)}
        if not self.attn_only:
            m.update({"wg": (F, H), "wu": (F, H), "wd": (H, F)})
        return m

    def params_per_layer(self) -> int:
        return sum(n * k for n, k in self.matrices().values())


SHAPES: Dict[str, ModelShape] = {
    # config 1: tiny single attention layer, bf16 weights
    "tiny": ModelShape("tiny", 256, 4, 1, 64, 0, 1, "bf16", attn_only=True),
    # config 2: Qwen2.5-7B shape, 28 layers, int4 g32
    "qwen7b": ModelShape("qwen7b", 3584, 28, 4, 128, 18944, 28, "int4"),
    # config 3: dense 9B-class verify shape
    "dense9b": ModelShape("dense9b", 4096, 32, 8, 128, 12288, 36, "int4"),
    # config 4: 4B-class prefix priming shape
    "dense4b": ModelShape("dense4b", 2560, 16, 8, 128, 9728, 36, "int4"),
    # config 5: one 7B-shaped attention + QKV/O layer
    "qwen7b_attn": ModelShape("qwen7b_attn", 3584, 28, 4, 128, 0, 1, "int4", attn_only=True),
    # small shapes for parity tests (several tiles, ragged tails)
    "small": ModelShape("small", 512, 8, 2, 64, 1024, 2, "int4"),
    "small_d128": ModelShape("small_d128", 768, 6, 2, 128, 768, 2, "int4"),
    "small_attn": ModelShape("small_attn", 512, 8, 2, 64, 0, 1, "int4", attn_only=True),
    "small_bf16": ModelShape("small_bf16", 256, 4, 2, 64, 512, 2, "bf16"),
    "small_q4k": ModelShape("small_q4k", 512, 8, 2, 64, 1024, 2, "q4k"),
    # head_dim 128 with four query heads per KV head (the small-m pass's shape class)
    "small_g4": ModelShape("small_g4", 512, 8, 2, 128, 1024, 3, "int4"),
    # hidden above 4096 (the row kernels' loops past the first 4096 elements of a row)
    "wide": ModelShape("wide", 4352, 8, 2, 64, 512, 1, "int4"),
    # the turn-9 and verify shapes with K-quant superblock weights
    "qwen7b_q4k": ModelShape("qwen7b_q4k", 3584, 28, 4, 128, 18944, 28, "q4k"),
    "dense9b_q4k": ModelShape("dense9b_q4k", 4096, 32, 8, 128, 12288, 36, "q4k"),
}


# ----------------------------------------------------------------------------
# bf16 inputs (torch's cast does the rounding; this is input preparation)
# ----------------------------------------------------------------------------

def to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def hidden_for_tokens(tokens: Sequence[int], hidden: int, seed: int) -> torch.Tensor:
    """bf16 [n][hidden]: row i is N(0,1) drawn from PCG64([seed, tokens[i]])."""
    rows = np.empty((len(tokens), hidden), dtype=np.float32)
    cache: Dict[int, np.ndarray] = {}
    for i, t in enumerate(tokens):
        t = int(t)
        if t not in cache:
            cache[t] = np.random.Generator(np.random.PCG64([seed, t])).standard_normal(hidden)
        rows[i] = cache[t]
    return to_bf16(rows)


# ----------------------------------------------------------------------------
# int4 group-32 weights
# ----------------------------------------------------------------------------

def _scale_up_5bit(s: torch.Tensor) -> torch.Tensor:
    """Round positive scales UP to 5 significant bits (then exact in fp16).

    A named extra case only: with such scales every code*scale has at most 8
    significant bits, a number both fp16 and bf16 hold exactly.
    """
    m, e = torch.frexp(s)                       # s = m * 2**e, m in [0.5, 1)
    m = torch.ceil(m * 32.0) / 32.0
    return torch.ldexp(m, e)


SCALES = ("fp16", "5bit")


def quantize_int4(w: torch.Tensor, scales: str = "fp16") -> tuple:
    """Symmetric int4 with one fp16 scale per 32 inputs.  w: float32 [N][K].

    Returns (codes int8 [N][K] in [-8, 7], scales fp16 [N][K/32]).
    scales="fp16" (the format as stated): scale = fp16(absmax / 7), round to
    nearest; scales="5bit": absmax / 7 rounded up to 5 significant bits.
    code = clamp(rne(w / scale), -8, 7) with the stored scale.
    """
    if scales not in SCALES:
        raise ValueError(f"scales must be one of {SCALES}")
    N, K = w.shape
    assert K % GROUP == 0
    g = w.reshape(N, K // GROUP, GROUP).to(torch.float32)
    amax = g.abs().amax(dim=-1)
    s = torch.clamp(amax / 7.0, min=2.0 ** -14)
    if scales == "5bit":
        s = _scale_up_5bit(s)
    s = s.to(torch.float16)
    q = torch.round(g / s.to(torch.float32).unsqueeze(-1)).clamp_(-8, 7).to(torch.int8)
    return q.reshape(N, K), s


def pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """Pack int8 codes [N][K] (values -8..7) into the kvr int4 byte layout.

    Each group of 32 inputs occupies 16 bytes = four little-endian 32-bit
    words.  Input k' (0..31 within the group) is stored as the 4-bit value
    k'-code + 8 in word (k' mod 8) div 2, nibble (k' div 8) + 4*(k' mod 2).
    Row n of the matrix is K/2 contiguous bytes.
    """
    N, K = codes.shape
    G = K // GROUP
    u = (codes.to(torch.int32) + 8)                        # 0..15
    # k' = 8a + 2w + b  ->  view as [N, G, a=4, w=4, b=2]
    u = u.reshape(N, G, 4, 4, 2)
    # nibble index nu = a + 4b within word w: order nibbles as (b, a)
    u = u.permute(0, 1, 3, 4, 2).reshape(N, G, 4, 8)        # [N, G, w, nu]
    lo = u[..., 0::2]                                      # nibble 2t  -> low half of byte t
    hi = u[..., 1::2]
    byte = (lo | (hi << 4)).to(torch.uint8)                # [N, G, w, 4 bytes]
    return byte.reshape(N, K // 2).contiguous()


@dataclasses.dataclass
class Int4Matrix:
    packed: torch.Tensor   # uint8 [N][K/2]
    scales: torch.Tensor   # fp16 [N][K/32]
    codes: Optional[torch.Tensor] = None  # int8 [N][K], kept only for small shapes


def make_int4(w: torch.Tensor, keep_codes: bool = False, scales: str = "fp16") -> Int4Matrix:
    q, s = quantize_int4(w, scales)
    return Int4Matrix(pack_int4(q), s.contiguous(), q if keep_codes else None)


# ----------------------------------------------------------------------------
# K-quant 4-bit superblocks (256 inputs: fp16 d and dmin, 6-bit scale and min
# per 32-input sub-block, unsigned 4-bit codes)
# ----------------------------------------------------------------------------

SUPER = 256


def _fp16_up(x: torch.Tensor) -> torch.Tensor:
    """Smallest fp16 value >= x (x >= 0), as float32."""
    h = x.to(torch.float16)
    low = h.to(torch.float32) < x
    h = torch.where(low, torch.nextafter(h, torch.full_like(h, float("inf"))), h)
    return h.to(torch.float32)


def quantize_q4k(w: torch.Tensor) -> tuple:
    """w float32 [N][K] -> (q uint [N][K] in [0, 15] as int8, d, dmin fp16 [N][K/256],
    sc, mn int [N][K/256][8] in [0, 63]).

    Per sub-block j: mn_j*dmin >= -min(w, 0) (every weight offset into [0, ...)),
    sc_j*d*15 >= the offset range, so rne((w + dmin*mn_j) / (d*sc_j)) lies in
    [0, 15] and the error is at most d*sc_j/2."""
    N, K = w.shape
    assert K % SUPER == 0
    g = w.reshape(N, K // SUPER, 8, GROUP).to(torch.float32)
    lo = torch.clamp(g.amin(dim=-1), max=0.0)
    hi = g.amax(dim=-1)
    dmin = _fp16_up(torch.clamp((-lo).amax(dim=-1) / 63.0, min=2.0 ** -24))
    mn = torch.clamp(torch.ceil(-lo / dmin.unsqueeze(-1)), 0, 63)
    off = mn * dmin.unsqueeze(-1)                          # exact: fp16 * small integer
    span = torch.clamp(hi + off, min=0.0) / 15.0
    d = _fp16_up(torch.clamp(span.amax(dim=-1) / 63.0, min=2.0 ** -24))
    sc = torch.clamp(torch.ceil(span / d.unsqueeze(-1)), 1, 63)
    step = (sc * d.unsqueeze(-1)).unsqueeze(-1)
    q = torch.round((g + off.unsqueeze(-1)) / step).clamp_(0, 15)
    return (q.to(torch.int8).reshape(N, K), d.to(torch.float16), dmin.to(torch.float16),
            sc.to(torch.int64), mn.to(torch.int64))


def pack_q4k_records(d: torch.Tensor, dmin: torch.Tensor, sc: torch.Tensor, mn: torch.Tensor) -> torch.Tensor:
    """uint8 [N][S*16]: per superblock fp16 d, fp16 dmin, then sixteen 6-bit
    fields (sc_0..7, mn_0..7), field f at bits 6f of a little-endian 96-bit string."""
    N, S = d.shape
    rec = torch.zeros((N, S, 16), dtype=torch.uint8, device=d.device)
    rec[..., 0:2] = d.contiguous().view(torch.uint8).reshape(N, S, 2)
    rec[..., 2:4] = dmin.contiguous().view(torch.uint8).reshape(N, S, 2)
    fields = torch.cat([sc, mn], dim=-1).to(torch.int64)  # [N, S, 16]
    # four fields per 24 bits -> 3 bytes
    f = fields.reshape(N, S, 4, 4)
    word = f[..., 0] | (f[..., 1] << 6) | (f[..., 2] << 12) | (f[..., 3] << 18)
    for b in range(3):
        rec[..., 4 + b::3][..., :4] = ((word >> (8 * b)) & 0xFF).to(torch.uint8)
    return rec.reshape(N, S * 16).contiguous()


@dataclasses.dataclass
class Q4KMatrix:
    packed: torch.Tensor   # uint8 [N][K/2]: the int4 nibble layout holding q in [0, 15]
    scales: torch.Tensor   # uint8 [N][K/256*16]: the superblock records


def make_q4k(w: torch.Tensor) -> Q4KMatrix:
    q, d, dmin, sc, mn = quantize_q4k(w)
    # pack_int4 stores code + 8: hand it q - 8
    return Q4KMatrix(pack_int4(q.to(torch.int16).sub(8).to(torch.int8)), pack_q4k_records(d, dmin, sc, mn))


# ----------------------------------------------------------------------------
# layer weights
# ----------------------------------------------------------------------------

_MAT_ORDER = ["wq", "wk", "wv", "wo", "wg", "wu", "wd"]


def norm_gain(hidden: int, seed: int, layer: int, which: int, device="cpu") -> torch.Tensor:
    """An RMSNorm gain: bf16 of U[0.5, 1.5) per element from PCG64([seed, layer,
    200 + which]) (which: 0 attention norm, 1 FFN norm, 2 the output head's),
    so a dropped, misplaced or swapped gain changes the result."""
    g = np.random.Generator(np.random.PCG64([seed, layer, 200 + which])).uniform(0.5, 1.5, hidden)
    return torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16).to(device)


def layer_weights(shape: ModelShape, seed: int, layer: int, device="cpu",
                  keep_codes: bool = False, std: float = 0.02, scales: str = "fp16") -> Dict[str, object]:
    """Weights of one layer.  bf16: tensors [N][K]; int4: Int4Matrix per matrix
    (scales: "fp16" or the named "5bit" case, see quantize_int4).

    Also 'norm_attn' and 'norm_ffn', the RMSNorm gains (norm_gain).
    """
    out: Dict[str, object] = {}
    for name, (n, k) in shape.matrices().items():
        idx = _MAT_ORDER.index(name)
        if str(device) == "cpu":
            rng = np.random.Generator(np.random.PCG64([seed, layer, idx]))
            w = torch.from_numpy(rng.standard_normal((n, k), dtype=np.float32) * np.float32(std))
        else:
            g = torch.Generator(device=device)
            g.manual_seed(seed * 1_000_003 + layer * 101 + idx)
            w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
        if shape.weight_format == "bf16":
            out[name] = w.to(torch.bfloat16).contiguous()
        elif shape.weight_format == "q4k":
            out[name] = make_q4k(w)
        else:
            out[name] = make_int4(w, keep_codes=keep_codes, scales=scales)
        del w
    H = shape.hidden
    if not shape.attn_only:
        out["norm_attn"] = norm_gain(H, seed, layer, 0, device)
        out["norm_ffn"] = norm_gain(H, seed, layer, 1, device)
    return out


def head_weights(shape: ModelShape, seed: int, device="cpu", vocab: int = VOCAB, keep_codes: bool = False,
                 std: float = 0.02) -> Dict[str, object]:
    """The output head: 'norm' (the final RMSNorm gain, norm_gain) and 'lm', the
    LM head [vocab][H] in the shape's weight format (int4 g32 or bf16)."""
    H = shape.hidden
    if str(device) == "cpu":
        rng = np.random.Generator(np.random.PCG64([seed, 10_000, 0]))
        w = torch.from_numpy(rng.standard_normal((vocab, H), dtype=np.float32) * np.float32(std))
    else:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1_000_003 + 10_000 * 101)
        w = torch.randn((vocab, H), generator=g, device=device, dtype=torch.float32) * std
    lm = w.to(torch.bfloat16).contiguous() if shape.weight_format == "bf16" else make_int4(w, keep_codes=keep_codes)
    return {"norm": norm_gain(H, seed, 10_000, 2, device), "lm": lm}


def stack_weights(shape: ModelShape, seed: int, device="cpu", keep_codes=False,
                  n_layers: Optional[int] = None, scales: str = "fp16") -> List[Dict[str, object]]:
    L = shape.n_layers if n_layers is None else n_layers
    return [layer_weights(shape, seed, l, device, keep_codes, scales=scales) for l in range(L)]


def weights_to(ws: List[Dict[str, object]], device) -> List[Dict[str, object]]:
    out = []
    for lw in ws:
        d = {}
        for k, v in lw.items():
            if isinstance(v, Int4Matrix):
                d[k] = Int4Matrix(v.packed.to(device), v.scales.to(device),
                                  None if v.codes is None else v.codes.to(device))
            elif isinstance(v, Q4KMatrix):
                d[k] = Q4KMatrix(v.packed.to(device), v.scales.to(device))
            else:
                d[k] = v.to(device)
        out.append(d)
    return out


# ----------------------------------------------------------------------------
# token lists of the five workloads
# ----------------------------------------------------------------------------

def config_seed(idx: int) -> int:
    return 1000 + idx


def fresh_tokens(rng: np.random.Generator, n: int, avoid_first: Optional[int] = None) -> List[int]:
    t = rng.integers(0, VOCAB, size=n).tolist()
    if avoid_first is not None and n > 0 and t[0] == avoid_first:
        t[0] = (avoid_first + 1) % VOCAB
    return t


def tiny_tokens(seed: int = config_seed(1)) -> Dict[str, List[int]]:
    """Config 1: slot0 = 96 tokens, slot1 = 64 tokens with another first token,
    prompt = slot0[:90] + 30 fresh tokens with prompt[90] != slot0[90]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    slot0 = fresh_tokens(rng, 96)
    slot1 = fresh_tokens(rng, 64, avoid_first=slot0[0])
    tail = fresh_tokens(rng, 30, avoid_first=slot0[90])
    return {"slot0": slot0, "slot1": slot1, "prompt": slot0[:90] + tail}


def turn9_tokens(seed: int = config_seed(2), template: int = 7,
                 prompt_len: int = 1922, cached: int = 1668,
                 slot0_len: int = 1700, others=(1500, 900, 300)) -> Dict[str, List[int]]:
    """Config 2: goinfer's turn-9 shape.  Every conversation starts with the same
    7-token chat-template prefix; slot0 holds the conversation whose first 1668
    tokens match the 1922-token prompt and then diverges; slots 1-3 hold other
    conversations that share only the template start."""
    rng = np.random.Generator(np.random.PCG64(seed))
    tmpl = fresh_tokens(rng, template)
    body = fresh_tokens(rng, cached - template)
    prompt_tail = fresh_tokens(rng, prompt_len - cached)
    slot0_tail = fresh_tokens(rng, slot0_len - cached, avoid_first=prompt_tail[0])
    prompt = tmpl + body + prompt_tail
    slot0 = tmpl + body + slot0_tail
    out = {"prompt": prompt, "slot0": slot0}
    for j, n in enumerate(others):
        rest = fresh_tokens(rng, n - template, avoid_first=body[0])
        out[f"slot{j + 1}"] = tmpl + rest
    return out


def verify_tokens(seed: int = config_seed(3), cached: int = 4096, max_rows: int = 8) -> Dict[str, List[int]]:
    rng = np.random.Generator(np.random.PCG64(seed))
    return {"state": fresh_tokens(rng, cached), "draft": fresh_tokens(rng, max_rows)}


def priming_tokens(seed: int = config_seed(4), state: int = 1200, n_q: int = 4,
                   q_len: int = 40) -> Dict[str, object]:
    rng = np.random.Generator(np.random.PCG64(seed))
    return {"state": fresh_tokens(rng, state),
            "questions": [fresh_tokens(rng, q_len) for _ in range(n_q)]}


def random_kv(n_kv_heads: int, n_tok: int, head_dim: int, seed: int) -> tuple:
    """Config 5: cached K/V drawn N(0,1) and rounded to bf16, [Hkv][n][d] each."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = rng.standard_normal((n_kv_heads, n_tok, head_dim), dtype=np.float32)
    v = rng.standard_normal((n_kv_heads, n_tok, head_dim), dtype=np.float32)
    return to_bf16(k), to_bf16(v)
