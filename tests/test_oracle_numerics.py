"""Pins of the oracle's numerics and weight decoding (no GPU)."""
import numpy as np
import torch

import workloads
from oracle import formats
from oracle.numerics import round_bf16, silu
from conftest import read_fixture


def test_round_bf16_matches_torch_cast(rng):
    # fp32-representable inputs: torch's fp32 -> bf16 cast is round-to-nearest-even
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_ties_to_even():
    # 1 + 2**-8 is halfway between 1 and 1 + 2**-7: ties to the even neighbour, 1
    assert round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2**-8 is halfway between 1+2**-7 (odd) and 1+2**-6 (even)
    assert round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # just above the tie rounds up; negative values are symmetric
    assert round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == -(1.0 + 2.0 ** -7)
    assert round_bf16(0.0) == 0.0
    # integers up to 256 are exact in bf16; 257 is a tie -> 256
    assert round_bf16(255.0) == 255.0 and round_bf16(257.0) == 256.0


def test_silu_identities(rng):
    x = rng.standard_normal(1000) * 5
    np.testing.assert_allclose(silu(x) - silu(-x), x, rtol=0, atol=1e-12)
    assert silu(0.0) == 0.0
    # sigmoid(1) = 1/(1+e^-1)
    np.testing.assert_allclose(silu(1.0), 0.7310585786300049, rtol=1e-15)


def test_int4_fixture_decodes():
    fx = read_fixture("int4_fixture.txt")
    packed = np.array([int(b, 16) for b in fx["bytes"]], dtype=np.uint8)[None, :]
    codes = np.array([int(c) for c in fx["codes"]])
    np.testing.assert_array_equal(formats.int4_codes(packed, 32)[0], codes)
    scales = np.array([[float(fx["scale"][0])]], dtype=np.float16)
    np.testing.assert_array_equal(formats.dequant_int4(packed, scales)[0], 0.5 * codes)


def test_packer_matches_fixture():
    fx = read_fixture("int4_fixture.txt")
    codes = torch.tensor([[int(c) for c in fx["codes"]]], dtype=torch.int8)
    got = workloads.pack_int4(codes).numpy()[0]
    np.testing.assert_array_equal(got, [int(b, 16) for b in fx["bytes"]])


def test_decode_inverts_pack(rng):
    q = torch.from_numpy(rng.integers(-8, 8, size=(37, 256)).astype(np.int8))
    packed = workloads.pack_int4(q).numpy()
    np.testing.assert_array_equal(formats.int4_codes(packed, 256), q.numpy().astype(np.int64))


def test_quantized_weights_are_exact_in_bf16(rng):
    # the synthetic quantiser's 5-bit scales make every code*scale a bf16 value
    w = torch.from_numpy(rng.standard_normal((64, 512)).astype(np.float32) * 0.02)
    m = workloads.make_int4(w)
    deq = formats.dequant_int4(m.packed.numpy(), m.scales.numpy())
    np.testing.assert_array_equal(round_bf16(deq), deq)
    # and the quantisation error is what int4 allows: |w - deq| <= scale/2
    s = m.scales.numpy().astype(np.float64).repeat(32, axis=1)
    assert np.all(np.abs(w.numpy() - deq) <= s / 2 + 1e-12)


def test_dequant_one_hot_column(rng):
    # x = e_k picks column k of W: pins the [N][K] orientation of the decoder
    q = torch.from_numpy(rng.integers(-8, 8, size=(8, 64)).astype(np.int8))
    s = torch.from_numpy((rng.uniform(0.5, 2, size=(8, 2))).astype(np.float16))
    W = formats.dequant_int4(workloads.pack_int4(q).numpy(), s.numpy())
    for k in (0, 5, 31, 32, 63):
        e = np.zeros(64); e[k] = 1.0
        np.testing.assert_array_equal(W @ e, q.numpy()[:, k] * s.numpy().astype(np.float64)[:, k // 32])


def test_bf16_bits_decode():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x3EAA], dtype=np.uint16)
    np.testing.assert_array_equal(formats.bf16_bits_to_f64(bits)[:3], [1.0, -2.0, 0.0])
    assert abs(formats.bf16_bits_to_f64(bits)[3] - 0.33203125) == 0
