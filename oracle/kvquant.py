"""FP8 (E4M3) KV cache, float64 oracle (test infrastructure only).

Not on the pages: their low-precision work (FlashDrive tutorial, quantisation
stage) concerns weights.  This is the KV-cache variant of the attention
operator: keys and values stored as 8-bit floats, E4M3 as the OCP 8-bit
floating-point format defines it (1 sign, 4 exponent bits with bias 7, 3
mantissa bits; exponent field 0 holds the subnormals m/8 * 2^-6; the pattern
S.1111.111 is NaN and there is no infinity, so the largest finite value is
448), with one power-of-two scale per (KV head, block of 128 cache rows):
the dequantised row r of head h is the E4M3 value times 2^exp[h, r // 128].

Readings: the block is 128 rows of the cache buffer (counted from its first
row), and the scale is a power of two, so that the dequantised value is exact
in bf16 and the attention over the dequantised cache is the same computation
as over a bf16 cache holding those values.
"""
from __future__ import annotations

import numpy as np

KV_BLOCK = 128


def e4m3_value(b: int) -> float:
    """The value of one E4M3 byte (NaN for S.1111.111)."""
    b = int(b) & 0xFF
    sign = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def dequantize(q8, exps) -> np.ndarray:
    """float64 [H, S, D] from E4M3 bytes q8 [H, S, D] (uint8) and block
    exponents exps [H, >= ceil(S / 128)] (int): q8 value * 2^exp[h, s // 128]."""
    q8 = np.asarray(q8, dtype=np.uint8)
    H, S, _ = q8.shape
    blocks = np.arange(S) // KV_BLOCK
    scale = np.ldexp(1.0, np.asarray(exps, dtype=np.int64)[:, blocks])      # [H, S]
    return E4M3_TABLE[q8] * scale[:, :, None]
