"""Evaluation bounds: how far another correct FP32 evaluation of the layer may lie
from the oracle (test infrastructure only, like the rest of the oracle).

The layer quantises FP32 values to E4M3 at several points ("DeepSeek-V3的MoE架构
设计革新" §2 FP8 training, items 1-2: activations per 1x128 tile, weights per
128x128 block, FP32 promotion per 128-element chunk). Two correct evaluations
of such a value -- the oracle's exact value rounded to FP32 and a device's
FP32 arithmetic -- differ by their rounding; where that difference spans a
rounding boundary of the E4M3 grid the two pick neighbouring codes, and the
dequantised operand then differs by a whole code step. The pages give no error
bound, so the bounds here are derived from the arithmetic:

* gemm_bound: an FP8 GEMM promoted per 128-element chunk, evaluated in FP32,
  lies within u * (CHUNK_ROUNDINGS * sum|terms| + sum over chunks of
  (|f P| + |acc|)) of the exact sum (u = 2^-24, first order). Inside a chunk
  the tensor core adds four K=32 steps of exact E4M3 products into an FP32
  accumulator; how a step aligns its 32 products is not documented, so each
  step may round up to four times on partial sums no larger than the chunk's
  sum of |terms|. The promotion rounds the chunk's scale product (|f P|) and
  its fused multiply-add into the running sum (|acc| after the chunk), both
  evaluated from the exact partial sums. Pinned against the device's
  FP32-output GEMMs by GPU tests, on layer-like operands and on random codes
  over the whole E4M3 range.
* elementwise FP32 chains (SiLU and its gradient) add a few ulps (ARITH_ULPS;
  FAST_ULPS for the forward's fast exponential and division), and first-order
  sensitivities carry input bounds through them.
* gate_err: the gates from router logits within ROUTER_LOGIT_ERR of exact
  (pinned against the device router by a GPU test).
* quant_range: for values with an error bound, the range of dequantised values
  an evaluation within the bound may produce under the 1x128 rule (the value
  and its tile's amax each at either end of their intervals).

A quantity computed linearly from quantised operands then has a "budget": the
ranges times the absolute coefficients they enter with. A device result is
held to the budget plus the tolerance of its own arithmetic.
"""
from __future__ import annotations

import numpy as np

from . import e4m3
from .quant import TILE, dequant_1x128, quant_1x128, tile_scale

U = 2.0 ** -24           # unit roundoff of FP32 (round to nearest)
CHUNK_ROUNDINGS = 16     # roundings inside one 128-element chunk: four K=32 tensor-core steps, each
                         # aligning 32 exact products into the accumulator (its internal alignment is
                         # not documented: four roundings of the step's sum of |terms| are allowed)
ARITH_ULPS = 8           # an elementwise FP32 chain with exp and division (SiLU, its gradient)
FAST_ULPS = 16           # the same with the fast exponential and division
ROUTER_LOGIT_ERR = 1e-5  # |router logit - exact| of a correct FP32 router at these widths


def gemm_bound(A, B) -> np.ndarray:
    """Bound on |FP32 chunk-promoted evaluation - exact| of A @ B for dequantised operands
    (the chunk scales folded into the values), contraction in chunks of 128:
    u * (CHUNK_ROUNDINGS * (|A| @ |B|) + sum_i |P_i| + sum_i |acc_i|), P_i chunk i's partial
    product, acc_i the running sum after it."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    acc = np.zeros((A.shape[0], B.shape[1]))
    run = np.zeros_like(acc)
    for c in range(0, A.shape[1], TILE):
        p = A[:, c:c + TILE] @ B[c:c + TILE]
        acc += p
        run += np.abs(p) + np.abs(acc)
    return U * (CHUNK_ROUNDINGS * (np.abs(A) @ np.abs(B)) + run)


def gate_err(s_sel) -> np.ndarray:
    """Bound on |g_k - exact| of the gates g = s / sum(s) for affinities s = sigmoid(z) whose
    logits are within ROUTER_LOGIT_ERR: |ds| <= err / 4 (sigmoid's slope), and
    dg_k = (ds_k - g_k sum_j ds_j) / S, plus two roundings."""
    s = np.asarray(s_sel, np.float64)
    S = s.sum(axis=1, keepdims=True)
    g = s / S
    ds = ROUTER_LOGIT_ERR / 4
    return ds * (1.0 + g * s.shape[1]) / S + 2 * U * g


def silu_derivs(a):
    """sigma(a), SiLU(a) = a sigma(a), SiLU'(a), SiLU''(a) in float64."""
    a = np.asarray(a, np.float64)
    sig = 1.0 / (1.0 + np.exp(-a))
    silu = a * sig
    d1 = sig * (1.0 + a * (1.0 - sig))
    d2 = sig * (1.0 - sig) * (2.0 + a * (1.0 - 2.0 * sig))
    return sig, silu, d1, d2


def tile_range(v, err, rule: str = "fp32"):
    """[lo, hi] per element of the dequantised values of v under the 1x128 rule along the
    last axis when each element may be off by up to err: the four corner evaluations, value
    low/high x tile amax low/high (the amax's own interval from every element's)."""
    v = np.asarray(v, np.float64)
    err = np.broadcast_to(np.asarray(err, np.float64), v.shape)
    rows, cols = v.shape
    t = v.reshape(rows, cols // TILE, TILE)
    et = err.reshape(rows, cols // TILE, TILE)
    # the tile amax of any evaluation within err lies in [max(|v| - err), max(|v| + err)]
    am_lo = np.maximum(np.abs(t) - et, 0.0).max(axis=2)
    am_hi = (np.abs(t) + et).max(axis=2)
    outs = []
    for vs in (t - et, t + et):
        for am in (am_lo, am_hi):
            sc = tile_scale(am.astype(np.float32), rule).astype(np.float64)
            scb = np.broadcast_to(sc[:, :, None], t.shape)
            with np.errstate(divide="ignore", invalid="ignore"):
                r = np.where(scb > 0, (vs / scb).astype(np.float32), np.float32(0.0))
            outs.append(e4m3.decode(e4m3.encode(r)) * scb)
    stack = np.stack(outs)
    return stack.min(axis=0).reshape(rows, cols), stack.max(axis=0).reshape(rows, cols)


def quant_range(v, err, rule: str = "fp32"):
    """(dequantised 1x128 quantisation of fl32(v), width of the range of dequantised values an
    evaluation within err of v may produce)."""
    v32 = np.asarray(v, np.float64).astype(np.float32)
    q, s = quant_1x128(v32, rule)
    deq = dequant_1x128(q, s)
    lo, hi = tile_range(v32, err, rule)
    return deq, np.maximum(hi, deq) - np.minimum(lo, deq)


def swiglu_h_bound(a, b, e_a, e_b, ulps: int = FAST_ULPS) -> np.ndarray:
    """Bound on |h - exact| of h = SiLU(a) * b evaluated in FP32 from a, b within e_a, e_b."""
    _, silu, d1, _ = silu_derivs(a)
    b = np.asarray(b, np.float64)
    return np.abs(d1 * b) * e_a + np.abs(silu) * e_b + ulps * U * np.abs(silu * b)
