"""Expert FFN on FP8 operands with fine-grained scales.

* Contraction: "DeepSeek-V3的MoE架构设计革新" §2 FP8 training, items 1-2. The
  product of an activation tile (scaled per 1x128) and a weight block
  (scaled per 128x128) is summed over each 128-element chunk of the
  contraction dimension and promoted to full precision with the two scales
  of that chunk:
      D[m, n] = sum_kc sa[m, kc] * sb[n // 128, kc] * sum_{k in kc} qa[m, k] qb[n, k]
  with qa, qb the decoded E4M3 values. Each chunk sum is exact in float64
  (products of E4M3 values are multiples of 2^-18 below 2^18).
* Expert: SwiGLU, W2 (SiLU(W1 u) * (W3 u)), the plain reading of the FFN
  the pages name; SiLU(g) = g * sigmoid(g). The intermediate h is rounded
  to float32 and quantised per 1x128 tile before the down projection (the
  activation rule applies to every FP8 GEMM input); the expert output is
  kept unrounded (the layer stores one rounded result, its output).
"""
from __future__ import annotations

import numpy as np

from . import e4m3
from .quant import TILE, quant_1x128, quant_128x128


def gemm_fp8(qa, sa, qb, sb, with_bound: bool = False):
    """qa u8 [m][k], sa f32 [m][k/128], qb u8 [n][k], sb f32 [n/128][k/128] -> float64 [m][n].

    with_bound: also return, per output, the bound on an FP32 evaluation's error
    (oracle/bounds.py, gemm_bound), from the same chunk partial sums."""
    A = e4m3.decode(qa)
    B = e4m3.decode(qb)
    m, k = A.shape
    n = B.shape[0]
    sa = np.asarray(sa, np.float64)
    sb = np.asarray(sb, np.float64)
    out = np.zeros((m, n), dtype=np.float64)
    if with_bound:
        from .bounds import CHUNK_ROUNDINGS, U
        absum = np.zeros((m, n), dtype=np.float64)
        run = np.zeros((m, n), dtype=np.float64)
    for kc in range(k // TILE):
        cols = slice(kc * TILE, (kc + 1) * TILE)
        partial = A[:, cols] @ B[:, cols].T
        col_scale = np.repeat(sb[:, kc], TILE)
        f = sa[:, kc][:, None] * col_scale[None, :]
        out += partial * f
        if with_bound:
            absum += (np.abs(A[:, cols]) @ np.abs(B[:, cols]).T) * np.abs(f)
            run += np.abs(partial * f) + np.abs(out)
    return (out, U * (CHUNK_ROUNDINGS * absum + run)) if with_bound else out


def silu(g):
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


def round_bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # below 2^-126 the spacing stays 2^-133
    q = np.round(np.ldexp(v, 8 - e))         # 8 significant bits, half to even
    return np.ldexp(q, e - 8)


class QuantExpert:
    """One expert's weights quantised per 128x128 block (scale rule `rule`, see quant)."""

    def __init__(self, w1, w3, w2, rule: str = "fp32"):
        self.rule = rule
        self.q1, self.s1 = quant_128x128(w1, rule)
        self.q3, self.s3 = quant_128x128(w3, rule)
        self.q2, self.s2 = quant_128x128(w2, rule)


def expert_forward(xq, xs, w: QuantExpert, return_h: bool = False, budget: bool = False):
    """xq u8 [m][d], xs f32 [m][d/128] -> float64 [m][d]; h is quantised by the expert's rule.

    budget: also return, per output element, how far another correct FP32 evaluation may
    lie from it through the E4M3 decision on h alone (oracle/bounds.py): the gate and up
    GEMMs' error bounds carried through SiLU, the resulting range of each dequantised h,
    and that range through |W2|."""
    if budget:
        from .bounds import swiglu_h_bound, tile_range
        from .quant import dequant_128x128
        gate, e_gate = gemm_fp8(xq, xs, w.q1, w.s1, with_bound=True)
        up, e_up = gemm_fp8(xq, xs, w.q3, w.s3, with_bound=True)
    else:
        gate = gemm_fp8(xq, xs, w.q1, w.s1)
        up = gemm_fp8(xq, xs, w.q3, w.s3)
    h = (silu(gate) * up).astype(np.float32)
    hq, hs = quant_1x128(h, w.rule)
    out = gemm_fp8(hq, hs, w.q2, w.s2)
    if budget:
        e_h = swiglu_h_bound(gate, up, e_gate, e_up)
        lo, hi = tile_range(h, e_h, w.rule)
        hd = e4m3.decode(hq).reshape(h.shape[0], -1, TILE) * np.asarray(hs, np.float64)[:, :, None]
        hd = hd.reshape(h.shape)
        delta_h = np.maximum(hi, hd) - np.minimum(lo, hd)
        return out, delta_h @ np.abs(dequant_128x128(w.q2, w.s2)).T
    if return_h:
        return out, h, hq, hs
    return out
