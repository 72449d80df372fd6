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
    """float32 values -> uint8 codes, round-to-nearest-even, saturating at 448.

    Rounds the magnitude a (clamped to 448) to a multiple of the E4M3 spacing
    of its binade, 2^(e-3) with e = max(floor(log2 a), -6); the multiple is
    chosen by round-half-to-even, which is the even-mantissa tie rule. The
    binade exponent is read from the float32 bit pattern; every division
    and product here is by a power of two, so it is exact.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.minimum(np.abs(v), np.float32(E4M3_MAX))
    e = ((a.view(np.uint32) >> 23).astype(np.int32) - 127)
    e = np.maximum(e, -6)
    spacing = ((e + (127 - 3)).astype(np.uint32) << 23).view(np.float32)
    r = np.round(a / spacing)                          # half to even
    val = r * spacing
    vb = val.view(np.uint32)
    normal = val >= np.float32(2.0 ** -6)
    exp_field = np.where(normal, (vb >> 23).astype(np.int32) - 127 + 7, 0)
    man_field = np.where(normal, (vb >> 20) & 7, r.astype(np.int32))
    code = (exp_field << 3) | man_field
    code = np.where(np.signbit(v), code | 0x80, code)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def encode_by_search(v) -> np.ndarray:
    """Same result as encode(), by nearest-neighbour search in the code table."""
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
