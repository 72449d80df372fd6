"""Backward pass of the DeepSeekMoE layer (test infrastructure only).

The pages frame the FP8 recipe as a training recipe ("DeepSeek-V3的MoE架构设计
革新" §2 FP8 training: activations per 1x128 tile, weights per 128x128
block, FP32 promotion every 128 elements of the contraction) and the
balancing as leaving the main loss's gradient untouched (《DeepSeek-V3
Technical Report》深度解读报告 §2.3: the bias acts on expert choice only).
They print no backward pass, so this module states the plain one:

* The layer is y = shared(x) + sum_k g_k(x) FFN_{e_k}(x), with the chosen
  experts e_k held fixed (choice is piecewise constant: no gradient flows
  through it, nor into the bias b).
* Gates: g_k = s_k / S, S = sum of the chosen s, s = sigmoid(z), z = x . Wr[e].
  dL/ds_j = (dg_j - sum_k g_k dg_k) / S for chosen j, dz_j = ds_j s_j (1 - s_j).
* SwiGLU: h = SiLU(a) b, SiLU(a) = a sigma(a).
  dA = dh b sigma(a) (1 + a (1 - sigma(a))), dB = dh SiLU(a).
* Every FP8 GEMM of the backward quantises its operands with the pages'
  rule for its operand kind, taken along the contracted dimension:
  - data gradients (dh = dO W2, dx = dA W1 + dB W3) quantise the gradient
    rows per 1x128 tile (like the forward's activations) and use the
    forward's 128x128-block weights, transposed (a block transposes exactly);
  - weight gradients (dW2 = dO^T h, dW1 = dA^T x, dW3 = dB^T x) contract
    over tokens, so both operands are quantised per 128 tokens x 1 channel
    ("128x1"), counted from the first row of each expert's rows (tokens in
    ascending order), the last tile of an expert zero-padded.
  Straight-through reading of quantisation: the operand of a weight
  gradient is the value the forward multiplied that weight with, i.e. the
  dequantised FP8 x and h (rounded to FP32, the product of an E4M3 value
  and an FP32 scale), re-tiled 128x1. Gradients enter as FP32 values:
  dO = fl32(g * dy) for routed rows and dy for the shared expert's rows,
  dA and dB rounded to FP32; the 1x128 tiles of a routed row's g * dy take
  dy's codes and scale fl32(g * s) under the FP32 rule (Quantiser.scaled_rows).

All arithmetic past those quantisation points is float64 on dequantised
values (the chunk-wise promotion of the GEMMs sums to the same value; see
ffn.gemm_fp8). With quantise=False every quantisation step is the identity
and the functions give the exact gradient of the float64 layer, which the
tests pin against finite differences.
"""
from __future__ import annotations

import numpy as np

from . import e4m3
from .ffn import silu
from .bounds import ARITH_ULPS, U, gate_err, gemm_bound, silu_derivs, swiglu_h_bound, tile_range
from .quant import TILE, dequant_1x128, quant_1x128


# ----------------------------------------------------------- quantisation ----
def segment_starts(offsets) -> np.ndarray:
    """Padded start column of each group's rows in a 128x1-tiled transposed
    operand: 128 * (number of 128-row tiles of the groups before it)."""
    offsets = np.asarray(offsets, np.int64)
    tiles = (np.diff(offsets) + TILE - 1) // TILE
    return np.concatenate([[0], np.cumsum(tiles) * TILE]).astype(np.int64)


def quant_128x1_grouped(v, offsets, rule: str = "fp32"):
    """v float32 [R][C] (rows grouped by `offsets` [G+1]) -> (qT u8 [C][Rp], sT f32 [Rp/128][C]).

    Group g's rows occupy columns P_g .. P_g + m_g - 1 of the transposed codes
    (P = segment_starts), zero-padded to a multiple of 128; each 128-column
    chunk of each row c of qT is one tile with its own scale sT[chunk][c]
    (the 1x128 rule applied along tokens). Padding codes are 0x00.
    """
    v = np.asarray(v, np.float32)
    offsets = np.asarray(offsets, np.int64)
    P = segment_starts(offsets)
    C = v.shape[1]
    qT = np.zeros((C, int(P[-1])), np.uint8)
    sT = np.zeros((int(P[-1]) // TILE, C), np.float32)
    for g in range(len(offsets) - 1):
        m = int(offsets[g + 1] - offsets[g])
        if m == 0:
            continue
        mp = int(P[g + 1] - P[g])
        seg = np.zeros((mp, C), np.float32)
        seg[:m] = v[offsets[g]:offsets[g + 1]]
        q, s = quant_1x128(np.ascontiguousarray(seg.T), rule)     # tiles of 128 tokens per channel
        qT[:, P[g]:P[g] + mp] = q
        sT[P[g] // TILE:P[g + 1] // TILE] = s.T
    return qT, sT


def dequant_128x1_grouped(qT, sT) -> np.ndarray:
    """Inverse layout of quant_128x1_grouped: float64 [C][Rp] values."""
    C, Rp = qT.shape
    return (e4m3.decode(qT).reshape(C, Rp // TILE, TILE)
            * np.asarray(sT, np.float64).T[:, :, None]).reshape(C, Rp)


def gemm_fp8_wgrad(qaT, saT, qbT, sbT) -> np.ndarray:
    """Weight-gradient contraction over tokens with 128x1 scales on both operands:
    D[m, n] = sum_kc saT[kc, m] * sbT[kc, n] * sum_{r in kc} qaT[m, r] qbT[n, r]  (float64)."""
    A = e4m3.decode(qaT)
    B = e4m3.decode(qbT)
    out = np.zeros((A.shape[0], B.shape[0]), np.float64)
    for kc in range(A.shape[1] // TILE):
        cols = slice(kc * TILE, (kc + 1) * TILE)
        out += (A[:, cols] @ B[:, cols].T) * (np.asarray(saT[kc], np.float64)[:, None]
                                              * np.asarray(sbT[kc], np.float64)[None, :])
    return out


def _fl32(v) -> np.ndarray:
    return np.asarray(v, np.float64).astype(np.float32)


# ------------------------------------------------------ evaluation bounds ----
# Two correct FP32 evaluations of the same gradient may straddle an E4M3
# rounding boundary (oracle/bounds.py). For each quantised operand the
# functions below carry a bound on how far a correct evaluation's input may
# lie from the oracle's ("err"), turn it into the range of dequantised values
# such an evaluation may produce ("delta"), and propagate the ranges linearly
# into "budgets" on the gradients.


class Quantiser:
    """The quantisation points of the backward; identity when `on` is False.

    Each call takes the values v (the oracle's, rounded to FP32 where the device stores FP32)
    and err, a bound on how far another correct evaluation's v may lie from them, and records
    in `delta` the width of the range of dequantised values such an evaluation may produce
    (zero where err is zero: the same bits on both sides)."""

    def __init__(self, rule: str = "fp32", on: bool = True):
        self.rule = rule
        self.on = on
        self.delta = None
        self.row_rel = None     # scaled_rows under the FP32 rule: the range is a uniform scaling per row

    def rows(self, v, err=0.0) -> np.ndarray:
        """1x128 tiles along the last axis (after rounding to FP32), dequantised."""
        if not self.on:
            self.delta = np.zeros(np.shape(v))
            return np.asarray(v, np.float64)
        v32 = _fl32(v)
        q, s = quant_1x128(v32, self.rule)
        deq = dequant_1x128(q, s)
        lo, hi = tile_range(v32, err, self.rule)
        self.delta = np.maximum(hi, deq) - np.minimum(lo, deq)
        return deq

    def scaled_rows(self, y, g, g_err=0.0) -> np.ndarray:
        """The 1x128 quantisation of g[i] * y[i] (g > 0 per row), dequantised; g may be off by g_err.

        FP32 rule: g scales each tile uniformly, so the codes are those of y's own tiles and
        the scale is fl32(g * s_y); a gate off by g_err moves every dequantised value by the
        same relative amount (no code changes). (Quantising fl32(g * y) again would leave
        the ratios 448 * y / max|y| -- often exact E4M3 midpoints for bf16 y -- to be
        decided by g's last bit.) Power-of-two rule: a power-of-two scale cannot absorb g,
        so fl32(g * y) is quantised, each value off by |y| * g_err.
        """
        y = np.asarray(y, np.float64)
        g = np.asarray(g, np.float64).reshape(-1, 1)
        ge = np.broadcast_to(np.asarray(g_err, np.float64).reshape(-1, 1) if np.ndim(g_err) else g_err, g.shape)
        if not self.on:
            self.delta = np.zeros(y.shape)
            return g * y
        if self.rule != "fp32":
            return self.rows(_fl32(g * y), np.abs(y) * ge + U * np.abs(g * y))
        q, s = quant_1x128(_fl32(y), self.rule)
        deq = dequant_1x128(q, (g * s.astype(np.float64)).astype(np.float32))
        self.row_rel = (2.0 * (ge / g + U)).ravel()       # every value of a row moves by this relative range
        self.delta = np.abs(deq) * self.row_rel[:, None]
        return deq

    def tokens(self, v, err=0.0) -> np.ndarray:
        """128x1 tiles along the first axis (one group of rows), dequantised: [m][C] float64."""
        if not self.on:
            self.delta = np.zeros(np.shape(v))
            return np.asarray(v, np.float64)
        v = _fl32(v)
        m, C = v.shape
        qT, sT = quant_128x1_grouped(v, [0, m], self.rule)
        deq = dequant_128x1_grouped(qT, sT)[:, :m].T
        mp = qT.shape[1]
        pad = np.zeros((mp, C))
        pad[:m] = v
        epad = np.zeros((mp, C))
        epad[:m] = np.broadcast_to(np.asarray(err, np.float64), v.shape)
        lo, hi = tile_range(pad.T, epad.T, self.rule)
        self.delta = (np.maximum(hi.T[:m], deq) - np.minimum(lo.T[:m], deq))
        return deq


# ------------------------------------------------------------- the pieces ----
def swiglu_grad(a, b, dh):
    """(dA, dB) of h = SiLU(a) * b for upstream dh (float64)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    dh = np.asarray(dh, np.float64)
    sig = 1.0 / (1.0 + np.exp(-a))
    return dh * b * sig * (1.0 + a * (1.0 - sig)), dh * silu(a)


def gate_grad(s_sel, dg):
    """Router logit gradient of the K chosen experts: s_sel, dg [T][K] -> dz [T][K]."""
    s_sel = np.asarray(s_sel, np.float64)
    dg = np.asarray(dg, np.float64)
    S = s_sel.sum(axis=1, keepdims=True)
    g = s_sel / S
    ds = (dg - (dg * g).sum(axis=1, keepdims=True)) / S
    return ds * s_sel * (1.0 - s_sel)


def expert_dgrad(xd, W1, W3, W2, dOd, Q: Quantiser, dOd_delta=None, dOd_row_rel=None) -> dict:
    """Rows of one expert: forward recomputation and data gradient.

    xd [m][d] the expert's input rows as the forward multiplied them (dequantised FP8; the
    same bits on every side); W1, W3 [I][d], W2 [d][I] the weights as the forward used them
    (dequantised blocks); dOd [m][d] the expert-output gradient as the data-gradient GEMM
    quantised it (Quantiser.scaled_rows), with either dOd_row_rel, the relative range of a
    whole row scaled uniformly (the FP32 rule: a gate error rescales the row, so dh moves by
    the same relative amount), or dOd_delta, the range of each dequantised value.

    With Q on, also the error bounds: e_a, e_b of the gate/up GEMM outputs, e_h of h (fast
    SiLU), e_dh of the dh GEMM (plus the gate's effect through dOd_delta), e_dA, e_dB by
    first-order sensitivities of the SwiGLU gradient, and the ranges delta_h, delta_dA,
    delta_dB of the quantised h, dA, dB; budget_dx = delta_dA @ |W1| + delta_dB @ |W3|.
    """
    a = xd @ W1.T
    b = xd @ W3.T
    sig, silu, d1, d2 = silu_derivs(a)
    h = silu * b
    d, I = xd.shape[1], W1.shape[0]
    if Q.on:
        e_a = gemm_bound(xd, W1.T)
        e_b = gemm_bound(xd, W3.T)
        e_h = swiglu_h_bound(a, b, e_a, e_b)
    else:
        e_a = e_b = e_h = np.zeros_like(a)
    hd = Q.rows(_fl32(h) if Q.on else h, e_h)
    delta_h = Q.delta
    out = hd @ W2.T
    dh = dOd @ W2
    if Q.on:
        e_dh = gemm_bound(dOd, W2)
        if dOd_row_rel is not None:
            e_dh = e_dh + dOd_row_rel[:, None] * np.abs(dh)
        elif dOd_delta is not None:
            e_dh = e_dh + dOd_delta @ np.abs(W2)
    else:
        e_dh = np.zeros_like(dh)
    dA, dB = swiglu_grad(a, b, dh)
    e_dA = np.abs(b * d1) * e_dh + np.abs(dh * d1) * e_b + np.abs(dh * b * d2) * e_a + ARITH_ULPS * U * np.abs(dA)
    e_dB = np.abs(silu) * e_dh + np.abs(dh * d1) * e_a + ARITH_ULPS * U * np.abs(dB)
    dAd = Q.rows(dA, e_dA)
    delta_dA = Q.delta
    dBd = Q.rows(dB, e_dB)
    delta_dB = Q.delta
    dx = dAd @ W1 + dBd @ W3
    budget_dx = delta_dA @ np.abs(W1) + delta_dB @ np.abs(W3)
    return {"a": a, "b": b, "hd": hd, "out": out, "dh": dh, "dA": dA, "dB": dB, "dx": dx,
            "e_dA": e_dA, "e_dB": e_dB, "delta_h": delta_h, "budget_dx": budget_dx}


def expert_wgrad(xd, hd, dO, dA, dB, Q: Quantiser, delta_h=None, e_dO=0.0, e_dA=0.0, e_dB=0.0):
    """Weight gradients of one expert over all its rows (token order): dW1 [I][d], dW3
    [I][d], dW2 [d][I], and their budgets from the 128x1 operands' ranges: x's codes and
    scales are the same bits on every side; dA, dB, dO enter with their error bounds; h
    enters as the forward's dequantised E4M3 values, whose own range is delta_h. With Q on,
    budgets["base"] bounds each gradient's own FP32 evaluation (gemm_bound over the
    expert's 128-token chunks): a correct device result lies within budget + base of these
    values, element by element."""
    xt = Q.tokens(xd)
    dAt = Q.tokens(dA, e_dA)
    rA = Q.delta
    dBt = Q.tokens(dB, e_dB)
    rB = Q.delta
    dOt = Q.tokens(dO, e_dO)
    rO = Q.delta
    ht = Q.tokens(hd, 0.0 if delta_h is None else delta_h)
    rh = Q.delta
    budgets = {"dW1": rA.T @ np.abs(xt), "dW3": rB.T @ np.abs(xt),
               "dW2": rO.T @ np.abs(ht) + np.abs(dOt).T @ rh}
    if Q.on:
        # the contraction's own FP32 evaluation over the expert's 128-token chunks
        budgets["base"] = {"dW1": gemm_bound(dAt.T, xt), "dW3": gemm_bound(dBt.T, xt),
                           "dW2": gemm_bound(dOt.T, ht)}
    return dAt.T @ xt, dBt.T @ xt, dOt.T @ ht, budgets


# -------------------------------------------------------------- the layer ----
def dequant_expert(w):
    """A QuantExpert's weights as the GEMMs use them: float64 W1, W3 [I][d], W2 [d][I]."""
    from .quant import dequant_128x128
    return dequant_128x128(w.q1, w.s1), dequant_128x128(w.q3, w.s3), dequant_128x128(w.q2, w.s2)


def layer_backward(cfg, x, dy, Wr, idx, s_sel, experts_w, tokens=(), wgrad_experts=(), router_experts=(),
                   Q: Quantiser | None = None, xd=None) -> dict:
    """Gradients of the layer for upstream dy, routing (idx, s_sel) held fixed.

    x, dy [T][d]; Wr [E][d]; idx [T][K]; s_sel [T][K] the chosen experts' raw
    affinities. experts_w(e) -> (W1, W3, W2) float64 as the GEMMs use them
    (e == E: the shared expert). Evaluates dx and dz for `tokens`, the expert
    weight gradients for `wgrad_experts`, and the router weight rows dWr[e]
    for `router_experts`. xd (optional) is x as the expert GEMMs see it; by
    default the 1x128-quantised x (or x itself when Q is off).

    "budget" (with Q on) holds, per gradient element, how far another correct
    evaluation may lie from these values through its quantisation decisions
    alone (see Quantiser and expert_dgrad): dx [tokens][d], dz and dg
    [tokens][K], dWr {e: [d]}; the expert weight gradients' budgets are the
    fourth entry of each dW[e]. Routing follows the gates' error bound
    (gate_err): h enters dg = dy . out, dg enters dz, dz enters dx and dWr.
    """
    Q = Quantiser() if Q is None else Q
    T, K = idx.shape
    E = cfg.E
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    idx = np.asarray(idx)
    s64 = np.asarray(s_sel, np.float64)
    gate = s64 / s64.sum(axis=1, keepdims=True)
    ge = gate_err(s64) if Q.on else np.zeros_like(gate)
    if xd is None:
        xd = Q.rows(x)
    tokens = np.asarray(sorted(set(int(t) for t in tokens)), np.int64)
    wgrad_experts = sorted(set(int(e) for e in wgrad_experts))
    router_experts = sorted(set(int(e) for e in router_experts))

    # (token, slot) pairs whose expert rows are evaluated: for dx/dz every slot of the
    # tokens asked for and of the tokens routed to a router expert; for wgrad every row
    # of the expert
    need_tok = set(tokens.tolist())
    for e in router_experts:
        need_tok |= set(np.nonzero((idx == e).any(axis=1))[0].tolist())
    pairs: dict[int, set] = {}
    for t in need_tok:
        for k in range(K):
            pairs.setdefault(int(idx[t, k]), set()).add((t, k))
    for e in wgrad_experts:
        if e == E:
            continue
        tt, kk = np.nonzero(idx == e)
        pairs.setdefault(e, set()).update(zip(tt.tolist(), kk.tolist()))
    shared_tok = set(need_tok) | (set(range(T)) if E in wgrad_experts else set())

    def dO_of(t, k):
        return _fl32(gate[t, k] * dy[t]) if Q.on else gate[t, k] * dy[t]

    dx_rows: dict = {}
    out_rows: dict = {}
    bdx_rows: dict = {}
    bdg_rows: dict = {}
    grads_w: dict = {}
    for e, prs in sorted(pairs.items()):
        prs = sorted(prs)                                   # token order = the expert's row order
        tt = np.array([p[0] for p in prs])
        kk = np.array([p[1] for p in prs])
        dO = np.stack([dO_of(t, k) for t, k in prs])
        dOd = Q.scaled_rows(dy[tt], gate[tt, kk], ge[tt, kk])
        uniform = Q.on and Q.rule == "fp32"
        W1, W3, W2 = experts_w(e)
        r = expert_dgrad(xd[tt], W1, W3, W2, dOd, Q, dOd_delta=None if uniform else Q.delta,
                         dOd_row_rel=Q.row_rel if uniform else None)
        bdg = (r["delta_h"] * np.abs(dy[tt] @ W2)).sum(axis=1)     # h's range through dg = dy . (h W2^T)
        for i, p in enumerate(prs):
            dx_rows[p] = r["dx"][i]
            out_rows[p] = r["out"][i]
            bdx_rows[p] = r["budget_dx"][i]
            bdg_rows[p] = bdg[i]
        if e in wgrad_experts:
            e_dO = np.abs(dy[tt]) * ge[tt, kk][:, None] + U * np.abs(dO)
            grads_w[e] = expert_wgrad(xd[tt], r["hd"], dO, r["dA"], r["dB"], Q, r["delta_h"], e_dO, r["e_dA"],
                                      r["e_dB"])
    if shared_tok:
        st = np.array(sorted(shared_tok))
        W1, W3, W2 = experts_w(E)
        dys = _fl32(dy[st]) if Q.on else dy[st]
        dOd = Q.rows(dys)                                   # dy itself: the same bits on every side
        r = expert_dgrad(xd[st], W1, W3, W2, dOd, Q)
        dx_shared = dict(zip(st.tolist(), r["dx"]))
        bdx_shared = dict(zip(st.tolist(), r["budget_dx"]))
        if E in wgrad_experts:
            grads_w[E] = expert_wgrad(xd[st], r["hd"], dys, r["dA"], r["dB"], Q, r["delta_h"], 0.0, r["e_dA"],
                                      r["e_dB"])
    else:
        dx_shared, bdx_shared = {}, {}

    nt = sorted(need_tok)
    dg = np.array([[dy[t] @ out_rows[(t, k)] for k in range(K)] for t in nt]).reshape(len(nt), K)
    dz_all = gate_grad(s64[nt], dg) if nt else np.zeros((0, K))
    # dz_k = s_k (1 - s_k) / S * sum_j (delta_kj - g_j) dg_j: a dg range maps through |delta_kj - g_j|
    bdg = np.array([[bdg_rows[(t, k)] for k in range(K)] for t in nt]).reshape(len(nt), K)
    if nt:
        sn, gn = s64[nt], gate[nt]
        Sn = sn.sum(axis=1, keepdims=True)
        jac = np.abs(np.eye(K)[None, :, :] - gn[:, None, :])                # [t][k][j]
        bdz_all = sn * (1.0 - sn) / Sn * np.einsum("tkj,tj->tk", jac, bdg)
    else:
        bdz_all = np.zeros((0, K))
    dz_of = dict(zip(nt, dz_all))
    dg_of = dict(zip(nt, dg))
    bdz_of = dict(zip(nt, bdz_all))
    bdg_of = dict(zip(nt, bdg))

    Wr = np.asarray(Wr, np.float64)
    dx = np.zeros((len(tokens), cfg.d))
    bdx = np.zeros((len(tokens), cfg.d))
    for i, t in enumerate(tokens.tolist()):
        v = dx_shared[t].copy()
        b = bdx_shared[t].copy()
        for k in range(K):
            v += dx_rows[(t, k)] + dz_of[t][k] * Wr[idx[t, k]]
            b += bdx_rows[(t, k)] + bdz_of[t][k] * np.abs(Wr[idx[t, k]])
        dx[i] = v
        bdx[i] = b
    dWr, bdWr = {}, {}
    for e in router_experts:
        acc = np.zeros(cfg.d)
        bacc = np.zeros(cfg.d)
        for t in np.nonzero((idx == e).any(axis=1))[0].tolist():
            k = int(np.nonzero(idx[t] == e)[0][0])
            acc += dz_of[t][k] * x[t]
            bacc += bdz_of[t][k] * np.abs(x[t])
        dWr[e] = acc
        bdWr[e] = bacc
    tl = tokens.tolist()
    return {"dx": dx, "tokens": tokens, "dz": np.array([dz_of[t] for t in tl]).reshape(len(tokens), K),
            "dg": np.array([dg_of[t] for t in tl]).reshape(len(tokens), K),
            "dW": grads_w, "dWr": dWr,
            "budget": {"dx": bdx, "dz": np.array([bdz_of[t] for t in tl]).reshape(len(tokens), K),
                       "dg": np.array([bdg_of[t] for t in tl]).reshape(len(tokens), K), "dWr": bdWr}}
