"""Fine-grained FP8 quantisation ("DeepSeek-V3的MoE架构设计革新" §2 FP8 training,
item 1: weights per 128x128 block, activations per 1x128 tile).

For each tile: amax = max |v|; scale = fl32(amax / 448); code =
E4M3_RNE_SATFINITE(fl32(v / scale)). fl32 is the IEEE single-precision
rounding of the exact quotient, which numpy float32 division gives. A tile
whose amax is zero stores scale 0 and codes 0x00 / 0x80 by sign. The value a
code stands for is decode(code) * scale.
"""
from __future__ import annotations

import numpy as np

from . import e4m3

TILE = 128


def _quant_tiles(v: np.ndarray, amax: np.ndarray, scale_per_elem: np.ndarray) -> np.ndarray:
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (v / scale_per_elem).astype(np.float32)
    r = np.where(scale_per_elem == 0, np.where(np.signbit(v), np.float32(-0.0), np.float32(0.0)), r)
    return e4m3.encode(r)


def quant_1x128(x) -> tuple[np.ndarray, np.ndarray]:
    """x [rows][cols] float32 (cols % 128 == 0) -> (codes u8 [rows][cols], scale f32 [rows][cols/128])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % TILE == 0
    t = x.reshape(rows, cols // TILE, TILE)
    amax = np.abs(t).max(axis=2)
    scale = (amax / np.float32(e4m3.E4M3_MAX)).astype(np.float32)
    q = _quant_tiles(t, amax, np.broadcast_to(scale[:, :, None], t.shape))
    return q.reshape(rows, cols), scale


def quant_128x128(w) -> tuple[np.ndarray, np.ndarray]:
    """w [rows][cols] float32 (both % 128 == 0) -> (codes u8 [rows][cols], scale f32 [rows/128][cols/128])."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert rows % TILE == 0 and cols % TILE == 0
    t = w.reshape(rows // TILE, TILE, cols // TILE, TILE)
    amax = np.abs(t).max(axis=(1, 3))
    scale = (amax / np.float32(e4m3.E4M3_MAX)).astype(np.float32)
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
