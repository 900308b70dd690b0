import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")


def read_fixture(name):
    """Parse a golden fixture: '#' comments, then 'key v1 v2 ...' lines."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def oracle_weights(shape, lw):
    """workloads layer weights -> the oracle's float64 matrices (decoded by the oracle)."""
    import torch
    from oracle import formats
    import workloads
    W = {}
    for name, v in lw.items():
        if isinstance(v, workloads.Int4Matrix):
            W[name] = formats.dequant_int4(v.packed.cpu().numpy(), v.scales.cpu().numpy())
        elif isinstance(v, workloads.Q4KMatrix):
            W[name] = formats.dequant_q4k(v.packed.cpu().numpy(), v.scales.cpu().numpy())
        else:
            W[name] = v.detach().cpu().to(torch.float64).numpy()
    return W


def oracle_dims(shape):
    from oracle.model import Dims
    return Dims(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                shape.attn_only, shape.rope_theta, shape.rms_eps)


@pytest.fixture
def rng():
    return np.random.Generator(np.random.PCG64(1234))
