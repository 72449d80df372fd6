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


NEAR_TOL = 3e-5


def near_midpoint(ratio, tol: float = NEAR_TOL) -> np.ndarray:
    """Elements whose quantisation ratio v / scale lies within tol (relative) of
    a rounding midpoint of the E4M3 grid: a perturbation of v that small may
    round it to the neighbouring code. The default tol covers two evaluations
    of the same gradient element whose GEMM sums were accumulated
    differently (an FP8 tensor-core chunk product may be summed with less
    than FP32's 24-bit precision before its promotion, the reason the pages
    give for promoting every 128 elements)."""
    r = np.abs(np.asarray(ratio, np.float64))
    r = np.minimum(r, e4m3.E4M3_MAX)
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.where(r > 0, r, 1.0))), -6)
    sp = np.ldexp(1.0, (e - 3).astype(np.int64))
    mid = (np.floor(r / sp) + 0.5) * sp
    return (r > 0) & (np.abs(r - mid) < tol * r)


class Quantiser:
    """The quantisation points of the backward; identity when `on` is False.

    Each call records in `near` the elements that sit within `tol` of an E4M3
    rounding midpoint while one E4M3 step of them is more than `sig` of the
    norm of their tile's row or column (the line the quantised values feed):
    where another correct FP32 evaluation of the same value may pick a
    neighbouring code that matters. near_rows / near_cols: any per row /
    column."""

    def __init__(self, rule: str = "fp32", on: bool = True, tol: float = NEAR_TOL, sig: float = 2e-3):
        self.rule = rule
        self.on = on
        self.tol = tol
        self.sig = sig
        self.near = None

    @property
    def near_rows(self):
        return self.near.any(axis=1)

    @property
    def near_cols(self):
        return self.near.any(axis=0)

    def _flag(self, v32, sc, deq, axis):
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(sc > 0, v32.astype(np.float64) / sc, 0.0)
        r = np.minimum(np.abs(ratio), e4m3.E4M3_MAX)
        with np.errstate(divide="ignore"):
            e = np.maximum(np.floor(np.log2(np.where(r > 0, r, 1.0))), -6)
        step = np.ldexp(1.0, (e - 3).astype(np.int64)) * sc          # one E4M3 step, in value units
        self.near_raw = near_midpoint(ratio, self.tol)
        self.step = step
        return self.near_raw & self.significant(step, deq, axis)

    def significant(self, step, deq, axis):
        """Steps larger than `sig` of the norm of their line (row: axis 1, column: axis 0) of deq."""
        norm = np.linalg.norm(deq, axis=axis, keepdims=True)
        return step > self.sig * np.where(norm > 0, norm, np.inf)

    def rows(self, v) -> np.ndarray:
        """1x128 tiles along the last axis (after rounding to FP32), dequantised."""
        if not self.on:
            self.near = np.zeros(np.shape(v), bool)
            self.near_raw, self.step = self.near, np.zeros(np.shape(v))
            return np.asarray(v, np.float64)
        v32 = _fl32(v)
        q, s = quant_1x128(v32, self.rule)
        deq = dequant_1x128(q, s)
        self.near = self._flag(v32, np.repeat(s, TILE, axis=1), deq, axis=1)
        return deq

    def scaled_rows(self, y, g) -> np.ndarray:
        """The 1x128 quantisation of g[i] * y[i] (g > 0 per row), dequantised.

        FP32 rule: g scales each tile uniformly, so the codes are those of y's
        own tiles and the scale is fl32(g * s_y). (Quantising fl32(g * y) again
        would leave the ratios 448 * y / max|y| -- often exact E4M3 midpoints
        for bf16 y -- to be decided by g's last bit.) Power-of-two rule: a
        power-of-two scale cannot absorb g, so fl32(g * y) is quantised.
        Nothing is flagged in the FP32 case: the codes come from y alone.
        """
        y = np.asarray(y, np.float64)
        g = np.asarray(g, np.float64).reshape(-1, 1)
        if not self.on or self.rule != "fp32":
            return self.rows(g * y if not self.on else _fl32(g * y))
        q, s = quant_1x128(_fl32(y), self.rule)
        self.near = np.zeros(y.shape, bool)
        return dequant_1x128(q, (g * s.astype(np.float64)).astype(np.float32))

    def tokens(self, v) -> np.ndarray:
        """128x1 tiles along the first axis (one group of rows), dequantised: [m][C] float64."""
        if not self.on:
            self.near = np.zeros(np.shape(v), bool)
            return np.asarray(v, np.float64)
        v = _fl32(v)
        m = v.shape[0]
        qT, sT = quant_128x1_grouped(v, [0, m], self.rule)
        deq = dequant_128x1_grouped(qT, sT)[:, :m].T
        sc = np.repeat(sT, TILE, axis=0)[:m]
        self.near = self._flag(v, sc, deq, axis=0)
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


def expert_dgrad(xd, W1, W3, W2, dO, Q: Quantiser, dO_exact: bool = False, dOd=None) -> dict:
    """Rows of one expert: forward recomputation and data gradient.

    xd [m][d] the expert's input rows as the forward multiplied them
    (dequantised FP8); W1, W3 [I][d], W2 [d][I] the weights as the forward used
    them (dequantised blocks); dO [m][d] the gradient of the expert output
    (dO_exact: its values are inputs, not computed, so never flagged); dOd,
    if given, is dO already quantised for the data gradient (Quantiser.scaled_rows).
    """
    a = xd @ W1.T
    b = xd @ W3.T
    hd = Q.rows(_fl32(silu(a) * b) if Q.on else silu(a) * b)
    # h elements near a rounding midpoint, with their E4M3 step (judged in expert_wgrad against
    # the token direction, along which they enter the W2 gradient)
    near_h = (Q.near_raw.copy(), Q.step.copy()) if Q.on else None
    near = Q.near_rows.copy()
    out = hd @ W2.T
    if dOd is None:
        dh = Q.rows(dO) @ W2
        if not dO_exact:             # dO = dy itself (shared expert): the same bits on every side
            near |= Q.near_rows
    else:
        dh = dOd @ W2
    dA, dB = swiglu_grad(a, b, dh)
    dAd = Q.rows(dA)
    near |= Q.near_rows
    dBd = Q.rows(dB)
    near |= Q.near_rows
    dx = dAd @ W1 + dBd @ W3
    # near: rows with a quantised element (h, dO, dA, dB) near a rounding midpoint (see Quantiser);
    # near_h: (near-midpoint mask, E4M3 step) of the elements of h
    return {"a": a, "b": b, "hd": hd, "out": out, "dh": dh, "dA": dA, "dB": dB, "dx": dx, "near": near,
            "near_h": near_h}


def expert_wgrad(xd, hd, dO, dA, dB, Q: Quantiser, near_h=None, dO_exact: bool = False):
    """Weight gradients of one expert over all its rows (token order):
    dW1 [I][d], dW3 [I][d], dW2 [d][I], and the flags of the gradient rows and
    columns fed by an operand channel with an element near a rounding
    midpoint (dA, dB, dO; h from near_h, the forward's own flags): a dict
    dW1 / dW3 -> rows [I], dW2 -> (rows [d], columns [I])."""
    xt = Q.tokens(xd)              # x's codes and scales are the same bits on both sides: no flags
    dAt = Q.tokens(dA)
    fA = Q.near_cols
    dBt = Q.tokens(dB)
    fB = Q.near_cols
    dOt = Q.tokens(dO)
    fO = Q.near_cols if not dO_exact else np.zeros(dO.shape[1], bool)
    ht = Q.tokens(hd)
    # h differs between evaluations: in its codes (near_h) and, through the tile scales of the
    # forward's 1x128 quantisation, in every dequantised value (the 128x1 requantisation's flags)
    fh = Q.near_cols.copy()
    if near_h is not None:
        raw, step = near_h
        fh |= (raw & Q.significant(step, hd, axis=0)).any(axis=0)
    flags = {"dW1": fA, "dW3": fB, "dW2": (fO, fh)}
    return dAt.T @ xt, dBt.T @ xt, dOt.T @ ht, flags


# -------------------------------------------------------------- the layer ----
def dequant_expert(w):
    """A QuantExpert's weights as the GEMMs use them: float64 W1, W3 [I][d], W2 [d][I]."""
    from .quant import dequant_128x128
    return dequant_128x128(w.q1, w.s1), dequant_128x128(w.q3, w.s3), dequant_128x128(w.q2, w.s2)


def layer_backward(cfg, x, dy, Wr, idx, s_sel, experts_w, tokens=(), wgrad_experts=(), router_experts=(),
                   Q: Quantiser | None = None, xd=None) -> dict:
    """Gradients of the layer for upstream dy, routing (idx, s_sel) held fixed.

    The result's "near" flags the tokens (of `tokens`) one of whose expert
    rows has a quantised element within Q.tol of an E4M3 rounding midpoint:
    there another correct FP32 evaluation may pick the neighbouring code.

    x, dy [T][d]; Wr [E][d]; idx [T][K]; s_sel [T][K] the chosen experts' raw
    affinities. experts_w(e) -> (W1, W3, W2) float64 as the GEMMs use them
    (e == E: the shared expert). Evaluates dx and dz for `tokens`, the expert
    weight gradients for `wgrad_experts`, and the router weight rows dWr[e]
    for `router_experts`. xd (optional) is x as the expert GEMMs see it; by
    default the 1x128-quantised x (or x itself when Q is off).
    """
    Q = Quantiser() if Q is None else Q
    T, K = idx.shape
    E = cfg.E
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    idx = np.asarray(idx)
    gate = np.asarray(s_sel, np.float64) / np.asarray(s_sel, np.float64).sum(axis=1, keepdims=True)
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
    near_tok: set = set()
    grads_w: dict = {}
    for e, prs in sorted(pairs.items()):
        prs = sorted(prs)                                   # token order = the expert's row order
        tt = np.array([p[0] for p in prs])
        kk = np.array([p[1] for p in prs])
        dO = np.stack([dO_of(t, k) for t, k in prs])
        dOd = Q.scaled_rows(dy[tt], gate[tt, kk])
        W1, W3, W2 = experts_w(e)
        r = expert_dgrad(xd[tt], W1, W3, W2, dO, Q, dOd=dOd)
        for i, p in enumerate(prs):
            dx_rows[p] = r["dx"][i]
            out_rows[p] = r["out"][i]
            if r["near"][i]:
                near_tok.add(p[0])
        if e in wgrad_experts:
            grads_w[e] = expert_wgrad(xd[tt], r["hd"], dO, r["dA"], r["dB"], Q, r["near_h"])
    if shared_tok:
        st = np.array(sorted(shared_tok))
        W1, W3, W2 = experts_w(E)
        r = expert_dgrad(xd[st], W1, W3, W2, dy[st] if not Q.on else _fl32(dy[st]), Q, dO_exact=True)
        dx_shared = dict(zip(st.tolist(), r["dx"]))
        near_tok |= set(st[r["near"]].tolist())
        if E in wgrad_experts:
            grads_w[E] = expert_wgrad(xd[st], r["hd"], _fl32(dy[st]) if Q.on else dy[st], r["dA"], r["dB"], Q,
                                      r["near_h"], dO_exact=True)
    else:
        dx_shared = {}

    nt = sorted(need_tok)
    dg = np.array([[dy[t] @ out_rows[(t, k)] for k in range(K)] for t in nt]).reshape(len(nt), K)
    dz_all = gate_grad(np.asarray(s_sel, np.float64)[nt], dg) if nt else np.zeros((0, K))
    dz_of = dict(zip(nt, dz_all))
    dg_of = dict(zip(nt, dg))

    Wr = np.asarray(Wr, np.float64)
    dx = np.zeros((len(tokens), cfg.d))
    for i, t in enumerate(tokens.tolist()):
        v = dx_shared[t].copy()
        for k in range(K):
            v += dx_rows[(t, k)] + dz_of[t][k] * Wr[idx[t, k]]
        dx[i] = v
    dWr = {}
    for e in router_experts:
        acc = np.zeros(cfg.d)
        for t in np.nonzero((idx == e).any(axis=1))[0].tolist():
            k = int(np.nonzero(idx[t] == e)[0][0])
            acc += dz_of[t][k] * x[t]
        dWr[e] = acc
    return {"dx": dx, "tokens": tokens, "dz": np.array([dz_of[t] for t in tokens.tolist()]).reshape(len(tokens), K),
            "dg": np.array([dg_of[t] for t in tokens.tolist()]).reshape(len(tokens), K),
            "dW": grads_w, "dWr": dWr,
            "near": np.array([t in near_tok for t in tokens.tolist()], bool)}
