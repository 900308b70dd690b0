"""Weight formats, decoded on the CPU.  Test infrastructure only.

int4 group-32 (the layout statement of ``include/kvr.h``):
    row n of a [N][K] matrix is K/2 bytes; group g of that row (inputs
    32g .. 32g+31) is the 16 bytes at offset 16g, read as four little-endian
    32-bit words.  Input k' = k - 32g is held in word (k' mod 8) div 2, in the
    4-bit field number (k' div 8) + 4*(k' mod 2) counted from the least
    significant bits; the field holds code + 8, code in [-8, 7].  The weight is
    code * scale[n][g], scale an fp16 number.

This module decodes that statement element by element, independently of the
packer in ``workloads``.  Pinned by: decode(pack(q)) == q for random q, and a
hand-written byte fixture (tests/golden/int4_fixture.txt).
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
