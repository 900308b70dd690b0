"""Scalar numerics of the oracle (float64).  Test infrastructure only.

round_bf16 -- round-to-nearest-even onto the bf16 grid (8 significant bits).
    Pinned: against torch's bf16 cast on fp32-representable values, and on
    hand-made ties (tests/test_oracle_numerics.py).
silu       -- x * sigmoid(x).  Pinned: silu(x) - silu(-x) == x, silu(0) == 0.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value of each float64 element, ties to even.

    bf16 keeps 8 significant bits: write x = f * 2**e with f in [0.5, 1),
    scale f to [128, 256), round that to the nearest integer (numpy's rint
    rounds halves to even) and scale back.  Valid for |x| within the bf16
    normal range, which covers every value this oracle produces; zero stays
    zero.
    """
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)


def silu(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))
