"""The small-m path defers RMSNorm past the projection (CPU only).

RMSNorm scales a row by one number r = rsqrt(mean(h^2) + eps), and a projection
is linear, so W (h r g) = r (W (h g)).  The GPU rounds h*g to bf16 and applies
r to the projection's fp32 result; the plain rounding point rounds h*r*g.
This checks, in float64 with the oracle's bf16 rounding, that both forms land
within the elementwise parity bound |x - ref| <= 1e-2 + 2e-2 |ref| of the exact
projection, with errors of the same size, at the full widths and at residual
stream scales from 1 to 30 (deep layers), for int4-like weights.
"""
import numpy as np
import pytest

from oracle import model as om
from oracle.numerics import round_bf16


@pytest.mark.parametrize("H,N,scale", [(3584, 512, 1.0), (4096, 512, 14.0), (2560, 512, 30.0)])
def test_deferred_norm_rounds_like_the_plain_rounding_point(H, N, scale):
    rng = np.random.default_rng(H + int(scale))
    h = rng.standard_normal((4, H)) * scale                         # residual rows
    g = round_bf16(1.0 + 0.1 * rng.standard_normal(H))              # RMSNorm gain (bf16)
    W = rng.integers(-8, 8, (N, H)) * round_bf16(np.full((N, 1), 0.02 / 7))   # code * scale
    eps = 1e-6
    r = 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    exact = om.rmsnorm(h, g, eps) @ W.T
    plain = round_bf16(om.rmsnorm(h, g, eps)) @ W.T                  # round the normed row
    deferred = (round_bf16(h * g) @ W.T) * r                         # round h*g, scale after
    bound = 1e-2 + 2e-2 * np.abs(exact)
    assert (np.abs(plain - exact) <= bound).all()
    assert (np.abs(deferred - exact) <= bound).all()
    e_plain = np.sqrt(np.mean((plain - exact) ** 2))
    e_def = np.sqrt(np.mean((deferred - exact) ** 2))
    assert 0.5 < e_def / e_plain < 2.0, (e_plain, e_def)             # the same size of error
