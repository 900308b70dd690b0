"""Weight formats, decoded on the CPU.  Test infrastructure only.

int4 group-32 (the layout statement of ``include/kvr.h``):
    row n of a [N][K] matrix is K/2 bytes; group g of that row (inputs
    32g .. 32g+31) is the 16 bytes at offset 16g, read as four little-endian
    32-bit words.  Input k' = k - 32g is held in word (k' mod 8) div 2, in the
    4-bit field number (k' div 8) + 4*(k' mod 2) counted from the least
    significant bits; the field holds code + 8, code in [-8, 7].  The weight is
    code * scale[n][g], scale an fp16 number.

K-quant 4-bit superblocks (KVR_WEIGHTS_Q4K; Tempo9 docs, "Models and
quantizations": Q4_K keeps 256 weights in 144 bytes, a superblock scale plus
per-sub-block scales and mins):
    the codes use the int4 nibble layout above, but a field holds q in [0, 15]
    with no offset; per row n and superblock s (inputs 256s .. 256s+255) a
    16-byte record at byte 16s of row n holds fp16 d (bytes 0-1), fp16 dmin
    (bytes 2-3) and a little-endian 96-bit string (bytes 4-15) of sixteen
    6-bit fields, field f at bits 6f: fields 0-7 the sub-block scales sc_j,
    fields 8-15 the mins mn_j, sub-block j = inputs 256s + 32j .. +31.  The
    weight is d*sc_j*q - dmin*mn_j.  128 + 16 = 144 bytes per 256 weights; the
    pages give that size only, so the layout inside is this library's.

This module decodes both statements element by element, independently of the
packers in ``workloads``.  Pinned by: decode(pack(q)) == q for random q, and
hand-written byte fixtures (tests/golden/int4_fixture.txt, q4k_fixture.txt).
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def int4_codes(packed: np.ndarray, K: int) -> np.ndarray:
    """uint8 [N][K/2] -> int64 codes [N][K] in [-8, 7]."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    assert packed.shape[1] * 2 == K and K % GROUP == 0
    words = packed.reshape(N, K // GROUP, 4, 4).astype(np.uint64)
    # little-endian 32-bit words: byte b has weight 256**b
    words = (words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24))
    codes = np.empty((N, K // GROUP, GROUP), dtype=np.int64)
    for kk in range(GROUP):
        w = (kk % 8) // 2
        field = kk // 8 + 4 * (kk % 2)
        codes[:, :, kk] = ((words[:, :, w] >> np.uint64(4 * field)) & np.uint64(0xF)).astype(np.int64) - 8
    return codes.reshape(N, K)


def dequant_int4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantised weight code * scale, float64 [N][K] (exact)."""
    scales = np.asarray(scales, dtype=np.float16).astype(np.float64)
    N, G = scales.shape
    K = G * GROUP
    codes = int4_codes(packed, K).astype(np.float64)
    return (codes.reshape(N, G, GROUP) * scales[:, :, None]).reshape(N, K)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (bf16 is the top half of fp32)."""
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(np.float64)


SUPER = 256


def q4k_record_fields(meta: np.ndarray):
    """uint8 [N][K/256*16] records -> (d, dmin) float64 [N][S] and (sc, mn) int64 [N][S][8]."""
    meta = np.asarray(meta, dtype=np.uint8)
    N = meta.shape[0]
    rec = meta.reshape(N, -1, 16)
    d = rec[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = rec[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    # the 96-bit string as an integer per record (byte b has weight 256**b)
    bits = [[int.from_bytes(bytes(rec[n, s, 4:16]), "little") for s in range(rec.shape[1])] for n in range(N)]
    fields = np.array([[[(x >> (6 * f)) & 63 for f in range(16)] for x in row] for row in bits],
                      dtype=np.int64).reshape(N, rec.shape[1], 16)
    return d, dmin, fields[..., :8], fields[..., 8:]


def dequant_q4k(packed: np.ndarray, meta: np.ndarray) -> np.ndarray:
    """Dequantised weight d*sc*q - dmin*mn, float64 [N][K] (exact: every term
    is a short product of fp16 numbers and small integers)."""
    packed = np.asarray(packed, dtype=np.uint8)
    N, K = packed.shape[0], packed.shape[1] * 2
    assert K % SUPER == 0
    q = (int4_codes(packed, K) + 8).astype(np.float64).reshape(N, K // SUPER, 8, GROUP)
    d, dmin, sc, mn = q4k_record_fields(meta)
    w = (d[:, :, None, None] * sc[:, :, :, None] * q) - (dmin[:, :, None, None] * mn[:, :, :, None])
    return w.reshape(N, K)
