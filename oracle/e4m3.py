"""E4M3 (FP8) codec written from the format definition.

Format ("DeepSeek-V3技术解析：MoE、FP8与MLA如何突破大模型推理瓶颈" §3.1: 4 exponent
bits, 3 mantissa bits; §6.2: the largest finite value is 448):

  code = s eeee mmm, exponent bias 7.
  eeee = 0     : subnormal, value = (-1)^s * m/8 * 2^(1-7)
  eeee = 1..15 : normal,    value = (-1)^s * (1 + m/8) * 2^(e-7)
  eeee = 15 and mmm = 7 is NaN (no infinities), so the top finite
  magnitude is 1.75 * 2^8 = 448.

Encoding rounds to the nearest representable value, ties to the code with
an even mantissa (round-to-nearest-even), and saturates anything at or
beyond 448 in magnitude to +-448 ("satfinite"). The sign of a value that
rounds to zero is kept (-0 is code 0x80).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _decode_code(c: int) -> float:
    s = -1.0 if (c >> 7) & 1 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


DECODE_TABLE = np.array([_decode_code(c) for c in range(256)], dtype=np.float64)

# Non-negative finite magnitudes in code order 0x00..0x7E (strictly increasing).
_POS = DECODE_TABLE[:0x7F].copy()


def decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(v) -> np.ndarray:
    """float32 values -> uint8 codes, round-to-nearest-even, saturating at 448."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    neg = np.signbit(v)
    a = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS, a, side="left")          # first magnitude >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS[hi] - a
    d_lo = a - _POS[lo]
    exact = d_hi == 0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(exact | pick_hi, hi, lo).astype(np.uint8)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    if np.isnan(v).any():
        code = np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)
    return code
