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
  dA and dB rounded to FP32.

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


class Quantiser:
    """The quantisation points of the backward; identity when `on` is False."""

    def __init__(self, rule: str = "fp32", on: bool = True):
        self.rule = rule
        self.on = on

    def rows(self, v) -> np.ndarray:
        """1x128 tiles along the last axis (after rounding to FP32), dequantised."""
        if not self.on:
            return np.asarray(v, np.float64)
        return dequant_1x128(*quant_1x128(_fl32(v), self.rule))

    def tokens(self, v) -> np.ndarray:
        """128x1 tiles along the first axis (one group of rows), dequantised: [m][C] float64."""
        if not self.on:
            return np.asarray(v, np.float64)
        v = _fl32(v)
        m = v.shape[0]
        qT, sT = quant_128x1_grouped(v, [0, m], self.rule)
        return dequant_128x1_grouped(qT, sT)[:, :m].T


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


def expert_dgrad(xd, W1, W3, W2, dO, Q: Quantiser) -> dict:
    """Rows of one expert: forward recomputation and data gradient.

    xd [m][d] the expert's input rows as the forward multiplied them
    (dequantised FP8); W1, W3 [I][d], W2 [d][I] the weights as the forward used
    them (dequantised blocks); dO [m][d] the gradient of the expert output.
    """
    a = xd @ W1.T
    b = xd @ W3.T
    hd = Q.rows(_fl32(silu(a) * b) if Q.on else silu(a) * b)
    out = hd @ W2.T
    dh = Q.rows(dO) @ W2
    dA, dB = swiglu_grad(a, b, dh)
    dx = Q.rows(dA) @ W1 + Q.rows(dB) @ W3
    return {"a": a, "b": b, "hd": hd, "out": out, "dh": dh, "dA": dA, "dB": dB, "dx": dx}


def expert_wgrad(xd, hd, dO, dA, dB, Q: Quantiser):
    """Weight gradients of one expert over all its rows (token order):
    dW1 [I][d], dW3 [I][d], dW2 [d][I]."""
    xt = Q.tokens(xd)
    return Q.tokens(dA).T @ xt, Q.tokens(dB).T @ xt, Q.tokens(dO).T @ Q.tokens(hd)


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
    grads_w: dict = {}
    for e, prs in sorted(pairs.items()):
        prs = sorted(prs)                                   # token order = the expert's row order
        tt = np.array([p[0] for p in prs])
        kk = np.array([p[1] for p in prs])
        dO = np.stack([dO_of(t, k) for t, k in prs])
        W1, W3, W2 = experts_w(e)
        r = expert_dgrad(xd[tt], W1, W3, W2, dO, Q)
        for i, p in enumerate(prs):
            dx_rows[p] = r["dx"][i]
            out_rows[p] = r["out"][i]
        if e in wgrad_experts:
            grads_w[e] = expert_wgrad(xd[tt], r["hd"], dO, r["dA"], r["dB"], Q)
    if shared_tok:
        st = np.array(sorted(shared_tok))
        W1, W3, W2 = experts_w(E)
        r = expert_dgrad(xd[st], W1, W3, W2, dy[st] if not Q.on else _fl32(dy[st]), Q)
        dx_shared = dict(zip(st.tolist(), r["dx"]))
        if E in wgrad_experts:
            grads_w[E] = expert_wgrad(xd[st], r["hd"], _fl32(dy[st]) if Q.on else dy[st], r["dA"], r["dB"], Q)
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
            "dW": grads_w, "dWr": dWr}
