"""Fine-grained FP8 quantisation ("DeepSeek-V3的MoE架构设计革新" §2 FP8 training,
item 1: weights per 128x128 block, activations per 1x128 tile).

For each tile: amax = max |v|; scale = fl32(amax / 448); code =
E4M3_RNE_SATFINITE(fl32(v / scale)). fl32 is the IEEE single-precision
rounding of the exact quotient, which numpy float32 division gives. A tile
whose amax is zero stores scale 0 and codes 0x00 / 0x80 by sign. The value a
code stands for is decode(code) * scale.

Power-of-two rule (rule="pow2", the block-scaled MX variant: the pages fix
the tile shapes and the 448 bound but not the scale's format, so this is a
second reading in which every scale has an 8-bit exponent code and no
mantissa): scale = the smallest power of two s with amax / s <= 448, but at
least 2^-126 (the smallest normal FP32 value); zero for an all-zero tile.
Then v / scale is exact (an exponent shift), |v / scale| <= 448, and the code
is E4M3_RNE(v / scale) as above.
"""
from __future__ import annotations

import numpy as np

from . import e4m3

TILE = 128


RULES = ("fp32", "pow2")
POW2_MIN_EXP = -126


def pow2_scale(amax) -> np.ndarray:
    """Smallest power of two s >= amax / 448 (i.e. 448 * s >= amax), at least 2^-126; 0 where amax == 0.

    amax lies in [2^k, 2^(k+1)) with k from frexp; 448 * 2^e >= amax then holds for
    e = k - 7 and fails for e = k - 9, so the answer is one of k - 9, k - 8, k - 7,
    each checked exactly in float64.
    """
    amax = np.asarray(amax, np.float64)
    out = np.zeros(amax.shape, np.float64)
    nz = amax > 0
    a = amax[nz]
    _, ex = np.frexp(a)                 # a = m * 2^ex, 0.5 <= m < 1
    k = ex - 1
    e = k - 7
    for cand in (k - 8, k - 9):
        e = np.where(448.0 * np.ldexp(1.0, cand) >= a, cand, e)
    e = np.maximum(e, POW2_MIN_EXP)
    out[nz] = np.ldexp(1.0, e)
    return out.astype(np.float32)


def tile_scale(amax, rule: str = "fp32") -> np.ndarray:
    """The scale of each tile from its amax under `rule`."""
    if rule == "fp32":
        return (np.asarray(amax, np.float32) / np.float32(e4m3.E4M3_MAX)).astype(np.float32)
    if rule == "pow2":
        return pow2_scale(amax)
    raise ValueError(f"rule: {rule!r}")


def _quant_tiles(v: np.ndarray, amax: np.ndarray, scale_per_elem: np.ndarray) -> np.ndarray:
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (v / scale_per_elem).astype(np.float32)
    r = np.where(scale_per_elem == 0, np.where(np.signbit(v), np.float32(-0.0), np.float32(0.0)), r)
    return e4m3.encode(r)


def quant_1x128(x, rule: str = "fp32") -> tuple[np.ndarray, np.ndarray]:
    """x [rows][cols] float32 (cols % 128 == 0) -> (codes u8 [rows][cols], scale f32 [rows][cols/128])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % TILE == 0
    t = x.reshape(rows, cols // TILE, TILE)
    amax = np.abs(t).max(axis=2)
    scale = tile_scale(amax, rule)
    q = _quant_tiles(t, amax, np.broadcast_to(scale[:, :, None], t.shape))
    return q.reshape(rows, cols), scale


def quant_128x128(w, rule: str = "fp32") -> tuple[np.ndarray, np.ndarray]:
    """w [rows][cols] float32 (both % 128 == 0) -> (codes u8 [rows][cols], scale f32 [rows/128][cols/128])."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert rows % TILE == 0 and cols % TILE == 0
    t = w.reshape(rows // TILE, TILE, cols // TILE, TILE)
    amax = np.abs(t).max(axis=(1, 3))
    scale = tile_scale(amax, rule)
    q = _quant_tiles(t, amax, np.broadcast_to(scale[:, None, :, None], t.shape))
    return q.reshape(rows, cols), scale


def dequant_1x128(q, scale) -> np.ndarray:
    rows, cols = q.shape
    return (e4m3.decode(q).reshape(rows, cols // TILE, TILE)
            * np.asarray(scale, np.float64)[:, :, None]).reshape(rows, cols)


def dequant_128x128(q, scale) -> np.ndarray:
    rows, cols = q.shape
    return (e4m3.decode(q).reshape(rows // TILE, TILE, cols // TILE, TILE)
            * np.asarray(scale, np.float64)[:, None, :, None]).reshape(rows, cols)
