"""Where the CUDA path rounds, measured against the elementwise bound (CPU only).

The bound is |x - ref| <= 1e-2 + 2e-2 |ref| on every element, residual stream
included.  This evaluates the FFN half of one full-width layer (the 4B-class
widths H = 2560, F = 9728, int4 group-32 weights with fp16 scales, residual
rows of rms 10 as in deep layers) in float32 with the GPU's rounding points,
and compares it with the same block in float64 with the oracle's (bf16 after
the RMSNorm and after SwiGLU, nothing else rounded):

* the small-m GEMV keeps each weight exact (code * scale in fp32) and rounds
  the normed row where the model does: its error is rounding noise;
* the tcgen05 GEMM rounds each weight once to fp16: larger, but well inside
  the bound;
* two forms the path used to take, rounding each weight to bf16 and deferring
  the RMSNorm factor past the projection (rounding h*g instead of h*r*g),
  each come close to the bound on these 2048 outputs and are several times
  the fp16 error, which is why neither is used.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats
from oracle import model as om
from oracle.numerics import round_bf16, silu

H, F, OUT = 2560, 9728, 512   # OUT: residual columns evaluated (all F inputs of the down projection)


def _int4(n, k, idx):
    """Exact int4 weights (code * fp16 scale) as float32, which holds them exactly."""
    rng = np.random.Generator(np.random.PCG64([5, idx]))
    w = torch.from_numpy(rng.standard_normal((n, k), dtype=np.float32) * np.float32(0.02))
    m = workloads.make_int4(w)
    return formats.dequant_int4(m.packed.numpy(), m.scales.numpy()).astype(np.float32)


@pytest.fixture(scope="module")
def block():
    Wg, Wu, Wd = _int4(F, H, 0), _int4(F, H, 1), _int4(OUT, F, 2)
    rng = np.random.Generator(np.random.PCG64(7))
    h = rng.standard_normal((4, H)) * 10.0
    g = round_bf16(rng.uniform(0.5, 1.5, H))
    return Wg, Wu, Wd, h, g


def _bf16_32(x):
    return round_bf16(np.asarray(x, dtype=np.float64)).astype(np.float32)


def _ffn_f64(Wg, Wu, Wd, h, g, eps=1e-6):
    b = round_bf16(om.rmsnorm(h, g, eps))
    gg, uu = b @ Wg.T.astype(np.float64), b @ Wu.T.astype(np.float64)
    return h[:, :OUT] + round_bf16(silu(gg) * uu) @ Wd.T.astype(np.float64)


def _ffn_f32(Wg, Wu, Wd, h, g, weights="exact", norm="plain", eps=1e-6):
    h32, g32 = h.astype(np.float32), g.astype(np.float32)
    r = (1.0 / np.sqrt(np.mean(h32 * h32, axis=-1, keepdims=True) + np.float32(eps))).astype(np.float32)
    if weights == "fp16":
        Wg, Wu, Wd = (w.astype(np.float16).astype(np.float32) for w in (Wg, Wu, Wd))
    elif weights == "bf16":
        Wg, Wu, Wd = (_bf16_32(w) for w in (Wg, Wu, Wd))
    if norm == "deferred":
        b = _bf16_32(h32 * g32)
        gg, uu = (b @ Wg.T) * r, (b @ Wu.T) * r
    else:
        b = _bf16_32(h32 * r * g32)
        gg, uu = b @ Wg.T, b @ Wu.T
    z = _bf16_32((gg / (np.float32(1) + np.exp(-gg))) * uu)
    return (h32[:, :OUT] + z @ Wd.T).astype(np.float64)


def _err(out, ref):
    err = np.abs(out - ref)
    return float((err / (1e-2 + 2e-2 * np.abs(ref))).max()), float(np.sqrt(np.mean(err ** 2)))


def test_rounding_points_against_the_elementwise_bound(block):
    ref = _ffn_f64(*block)
    gemv, gemv_rms = _err(_ffn_f32(*block), ref)
    gemm, gemm_rms = _err(_ffn_f32(*block, weights="fp16"), ref)
    bf16w, bf16w_rms = _err(_ffn_f32(*block, weights="bf16"), ref)
    deferred, deferred_rms = _err(_ffn_f32(*block, norm="deferred"), ref)
    print(f"max err / bound: exact weights {gemv:.4f}, fp16 weights {gemm:.3f}, "
          f"bf16 weights {bf16w:.3f}, deferred norm {deferred:.3f}")
    assert gemv < 0.02                     # rounding noise only
    assert gemm < 0.5                      # fp16 weights: inside the bound with margin
    assert bf16w > 0.6 and deferred > 0.6  # the rejected forms: near the bound already
    assert bf16w_rms > 2.5 * gemm_rms and deferred_rms > 2.5 * gemm_rms


# ----------------------------------------------------------------------------
# one whole 7B-width layer: the rounding points cascade
# ----------------------------------------------------------------------------
# Each bf16 rounding point (q/k/v, the attention output o, the normed rows,
# the SwiGLU product z) turns a perturbation far below one bf16 step into
# one-step flips with probability ~ perturbation / step, and every flip
# perturbs the next stage: a float32 evaluation differs from float64 in 0.5 %
# of o, ~1 % of the normed rows and ~15 % of z, and z feeds an 18944-input
# down projection.  At this width the residual stream (rms ~3) therefore
# carries errors of a few 1e-3 from float32 arithmetic alone, near an
# absolute 1e-2 per element; the residual rows of the full-size parity tests
# take the same bound with its absolute term in units of the row's rms.

H7, F7, HQ7, HKV7, D7, P7, M7 = 3584, 18944, 28, 4, 128, 1668, 8


@pytest.fixture(scope="module")
def layer7b():
    def mat(n, k, idx):
        rng = np.random.Generator(np.random.PCG64([11, idx]))
        w = torch.from_numpy(rng.standard_normal((n, k), dtype=np.float32) * np.float32(0.02))
        m = workloads.make_int4(w)
        return formats.dequant_int4(m.packed.numpy(), m.scales.numpy()).astype(np.float32)
    W32 = {"wq": mat(HQ7 * D7, H7, 0), "wk": mat(HKV7 * D7, H7, 1), "wv": mat(HKV7 * D7, H7, 2),
           "wo": mat(H7, HQ7 * D7, 3), "wg": mat(F7, H7, 4), "wu": mat(F7, H7, 5), "wd": mat(H7, F7, 6),
           "norm_attn": workloads.norm_gain(H7, 11, 0, 0).float().numpy(),
           "norm_ffn": workloads.norm_gain(H7, 11, 0, 1).float().numpy()}
    kk, vv = workloads.random_kv(HKV7, P7, D7, 12)
    x = workloads.bf16_to_f64(workloads.hidden_for_tokens(list(range(100, 100 + M7)), H7, 13))
    return W32, workloads.bf16_to_f64(kk), workloads.bf16_to_f64(vv), x


def _layer_f32(W32, Kp, Vp, x, rows, bf16_p):
    """The decoder layer in float32 with the oracle's rounding points; with
    bf16_p the softmax numerators enter the P V product rounded to bf16 (the
    row sum keeps their float32 values), as the tensor-core attention does."""
    G = HQ7 // HKV7
    h = x.astype(np.float32)

    def norm(v, g):
        r = (1.0 / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + np.float32(1e-6))).astype(np.float32)
        return _bf16_32(v * r * g)

    a = norm(h, W32["norm_attn"])
    k = (a @ W32["wk"].T).reshape(-1, HKV7, D7)
    v = (a @ W32["wv"].T).reshape(-1, HKV7, D7)
    K = np.zeros((HKV7, P7 + M7, D7), np.float32)
    V = np.zeros_like(K)
    K[:, :P7], V[:, :P7] = Kp, Vp
    for i, r in enumerate(rows):
        K[:, r.store] = _bf16_32(om.rope(k[i].astype(np.float64), r.pos, 1e6))
        V[:, r.store] = _bf16_32(v[i])
    q = (a @ W32["wq"].T).reshape(-1, HQ7, D7)
    o = np.empty((M7, HQ7, D7), np.float32)
    for i, r in enumerate(rows):
        qq = _bf16_32(om.rope(q[i].astype(np.float64), r.pos, 1e6))
        for hh in range(HQ7):
            s = (K[hh // G, r.visible] @ qq[hh]) / np.float32(np.sqrt(D7))
            e = np.exp(s - s.max()).astype(np.float32)
            o[i, hh] = ((_bf16_32(e) if bf16_p else e) @ V[hh // G, r.visible]) / e.sum()
    hs = h + _bf16_32(o).reshape(M7, -1) @ W32["wo"].T
    b = norm(hs, W32["norm_ffn"])
    g, u = b @ W32["wg"].T, b @ W32["wu"].T
    z = _bf16_32(g / (np.float32(1) + np.exp(-g)) * u)
    return (hs + z @ W32["wd"].T).astype(np.float64)


def test_full_width_layer_cascade(layer7b):
    W32, Kp, Vp, x = layer7b
    W = {k: v.astype(np.float64) for k, v in W32.items()}
    dims = om.Dims(H7, HQ7, HKV7, D7, F7, False, 1e6, 1e-6)
    rows = om.plain_rows(P7, M7)
    K = np.zeros((HKV7, P7 + M7, D7))
    V = np.zeros_like(K)
    K[:, :P7], V[:, :P7] = Kp, Vp
    ref = om.layer_rows(dims, W, x, K, V, rows, list(range(M7)))
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    plain, scaled = {}, {}
    for bf16_p in (False, True):
        err = np.abs(_layer_f32(W32, Kp, Vp, x, rows, bf16_p) - ref)
        plain[bf16_p] = err / (1e-2 + 2e-2 * np.abs(ref))
        scaled[bf16_p] = float((err / (1e-2 * rms + 2e-2 * np.abs(ref))).max())
    print(f"exact P: plain {plain[False].max():.3f} scaled {scaled[False]:.3f}; "
          f"bf16 P: plain {plain[True].max():.3f} ({int((plain[True] > 1).sum())} over) scaled {scaled[True]:.3f}")
    assert plain[False].max() > 0.5        # float32 arithmetic alone uses most of an absolute 1e-2
    assert (plain[True] > 1).sum() > 0     # with bf16 P (the tensor cores' operand) some elements exceed it
    assert scaled[False] < 0.5 and scaled[True] < 0.8   # the rms-scaled form holds with margin
