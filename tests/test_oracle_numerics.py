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


def test_quantizer_scales_and_error(rng):
    # the format as stated: scale = absmax/7 rounded to the nearest fp16
    # (numpy's own float16 cast pins the rounding), codes within [-8, 7], and
    # the quantisation error is what int4 allows: |w - deq| <= scale/2
    w = torch.from_numpy(rng.standard_normal((64, 512)).astype(np.float32) * 0.02)
    m = workloads.make_int4(w)
    amax = np.abs(w.numpy().reshape(64, 16, 32)).max(axis=-1)
    np.testing.assert_array_equal(m.scales.numpy(), (amax / np.float32(7.0)).astype(np.float16))
    deq = formats.dequant_int4(m.packed.numpy(), m.scales.numpy())
    s = m.scales.numpy().astype(np.float64).repeat(32, axis=1)
    assert np.all(np.abs(w.numpy() - deq) <= s / 2 + 1e-12)
    # general fp16 scales carry up to 11 significant bits: some code*scale is
    # not a bf16 number (the case the projections must handle exactly)
    assert np.any(round_bf16(deq) != deq)


def test_five_bit_scales_give_bf16_weights(rng):
    # the named extra case: scales rounded up to 5 significant bits make every
    # code*scale exactly a bf16 (and fp16) number
    w = torch.from_numpy(rng.standard_normal((64, 512)).astype(np.float32) * 0.02)
    m = workloads.make_int4(w, scales="5bit")
    deq = formats.dequant_int4(m.packed.numpy(), m.scales.numpy())
    np.testing.assert_array_equal(round_bf16(deq), deq)
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


# ---------------------------------------------------------------- K-quant superblocks

def _q4k_fixture():
    fx = read_fixture("q4k_fixture.txt")
    group = [int(b, 16) for b in fx["group"]]
    packed = np.array(group * 8, dtype=np.uint8)[None, :]
    record = np.array([int(b, 16) for b in fx["record"]], dtype=np.uint8)[None, :]
    return fx, packed, record


def test_q4k_fixture_decodes():
    fx, packed, record = _q4k_fixture()
    d, dmin, sc, mn = formats.q4k_record_fields(record)
    assert d[0, 0] == float(fx["d"][0]) and dmin[0, 0] == float(fx["dmin"][0])
    np.testing.assert_array_equal(sc[0, 0], [int(v) for v in fx["sc"]])
    np.testing.assert_array_equal(mn[0, 0], [int(v) for v in fx["mn"]])
    w = formats.dequant_q4k(packed, record)[0]
    for kv in fx["worked"]:
        k, v = kv.split(":")
        assert w[int(k)] == float(v), k


def test_q4k_packer_matches_fixture():
    fx, packed, record = _q4k_fixture()
    d = torch.tensor([[float(fx["d"][0])]], dtype=torch.float16)
    dmin = torch.tensor([[float(fx["dmin"][0])]], dtype=torch.float16)
    sc = torch.tensor([[[int(v) for v in fx["sc"]]]])
    mn = torch.tensor([[[int(v) for v in fx["mn"]]]])
    np.testing.assert_array_equal(workloads.pack_q4k_records(d, dmin, sc, mn).numpy(), record)
    q = torch.tensor([[k % 16 for k in range(256)]], dtype=torch.int16)
    np.testing.assert_array_equal(workloads.pack_int4((q - 8).to(torch.int8)).numpy(), packed)


def test_q4k_with_unit_scales_and_mins_of_eight_is_int4(rng):
    # sc = 1, mn = 8, d = dmin = s gives s*q - 8s = s*(q - 8): the int4 decode of
    # the same code bytes with scale s on every group of the superblock
    N, S = 5, 2
    packed = rng.integers(0, 256, size=(N, S * 128), dtype=np.uint8)
    s = rng.uniform(0.01, 0.1, size=(N, S)).astype(np.float16)
    bits = sum(1 << (6 * f) for f in range(8)) + sum(8 << (6 * f) for f in range(8, 16))
    tail = np.frombuffer(bits.to_bytes(12, "little"), dtype=np.uint8)
    record = np.zeros((N, S, 16), dtype=np.uint8)
    record[..., 0:2] = s.view(np.uint8).reshape(N, S, 2)
    record[..., 2:4] = s.view(np.uint8).reshape(N, S, 2)
    record[..., 4:] = tail
    got = formats.dequant_q4k(packed, record.reshape(N, S * 16))
    want = formats.dequant_int4(packed, np.repeat(s, 8, axis=1))
    np.testing.assert_array_equal(got, want)


def test_q4k_single_field_lands_on_its_sub_block():
    # one non-zero 6-bit field f: a scale (f < 8) scales sub-block f, a min
    # (f >= 8) offsets sub-block f - 8; every other sub-block decodes to 0
    packed = np.full((1, 128), 0x11, dtype=np.uint8)          # q = 1 everywhere
    for f in range(16):
        record = np.zeros((1, 16), dtype=np.uint8)
        record[0, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
        record[0, 2:4] = np.array([1.0], dtype=np.float16).view(np.uint8)
        record[0, 4:] = np.frombuffer((37 << (6 * f)).to_bytes(12, "little"), dtype=np.uint8)
        w = formats.dequant_q4k(packed, record)[0].reshape(8, 32)
        want = np.zeros((8, 32))
        want[f % 8] = 37.0 if f < 8 else -37.0
        np.testing.assert_array_equal(w, want, err_msg=f"field {f}")


def test_q4k_quantizer_error_bound(rng):
    w = torch.from_numpy(rng.standard_normal((16, 512)).astype(np.float32) * 0.02)
    m = workloads.make_q4k(w)
    deq = formats.dequant_q4k(m.packed.numpy(), m.scales.numpy())
    d, dmin, sc, mn = formats.q4k_record_fields(m.scales.numpy())
    step = (d[:, :, None] * sc).repeat(32, axis=-1).reshape(16, 512)
    assert np.all(np.abs(w.numpy() - deq) <= step / 2 * (1 + 1e-6) + 1e-12)
    assert sc.max() <= 63 and mn.max() <= 63 and sc.min() >= 1
