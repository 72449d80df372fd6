"""Router: sigmoid affinity, aux-loss-free group-limited top-K, gates.

Follows 《DeepSeek-V3 Technical Report》深度解读报告:

* §2.2 DeepSeekMoE: affinity s = sigmoid(u . e_i) (here z = x . Wr[i], plus an
  optional synthetic per-expert logit offset used only to skew a workload);
  gates are the affinities of the chosen experts renormalised to sum to 1.
* §2.3 Auxiliary-Loss-Free Load Balancing: the bias b_i is added to s_i only
  to choose experts; gates use the raw s_i.
* §2.4 Node-Limited Routing: a token may reach at most M groups, the groups
  ranked by the sum of the highest biased affinities of their experts (the
  gk largest, gk = K / M in every workload here).

Readings where the page is silent: groups are contiguous blocks of E/G
experts; group scores use the biased affinity (choosing groups is part of
choosing experts); equal scores are ordered by lower index; the K chosen
experts are listed by descending biased affinity.
"""
from __future__ import annotations

import numpy as np


def affinity(x, Wr, logit_offset=None) -> np.ndarray:
    """x [T][d], Wr [E][d] -> s = sigmoid(x Wr^T + o) in float64 [T][E]."""
    z = np.asarray(x, np.float64) @ np.asarray(Wr, np.float64).T
    if logit_offset is not None:
        z = z + np.asarray(logit_offset, np.float64)[None, :]
    return 1.0 / (1.0 + np.exp(-z))


def select(s, bias, G: int, M: int, K: int, gk: int):
    """Group-limited top-K on biased affinities.

    Returns (idx int32 [T][K], gate float64 [T][K], info) where info holds,
    per token, the margin between the M-th and (M+1)-th group scores and
    between the K-th chosen and the best unchosen expert of the kept groups
    (inf where no competitor exists), plus the smallest gap between
    consecutive chosen experts.
    """
    s = np.asarray(s, np.float64)
    T, E = s.shape
    n = E // G
    assert n * G == E and 1 <= M <= G and 1 <= gk <= n and K <= M * n
    sb = s + np.asarray(bias, np.float64)[None, :]

    # group score: sum of the gk largest biased affinities of the group
    grp = sb.reshape(T, G, n)
    top = -np.sort(-grp, axis=2)[:, :, :gk]
    gscore = top.sum(axis=2)
    gorder = np.argsort(-gscore, axis=1, kind="stable")      # desc, ties -> lower index
    keep = np.zeros((T, G), dtype=bool)
    np.put_along_axis(keep, gorder[:, :M], True, axis=1)

    masked = np.where(np.repeat(keep, n, axis=1), sb, -np.inf)
    eorder = np.argsort(-masked, axis=1, kind="stable")
    idx = eorder[:, :K].astype(np.int32)

    chosen = np.take_along_axis(s, idx, axis=1)
    gate = chosen / chosen.sum(axis=1, keepdims=True)

    gs = np.take_along_axis(gscore, gorder, axis=1)
    group_gap = gs[:, M - 1] - gs[:, M] if M < G else np.full(T, np.inf)
    ms = np.take_along_axis(masked, eorder, axis=1)
    if K < M * n:
        expert_gap = ms[:, K - 1] - ms[:, K]
    else:
        expert_gap = np.full(T, np.inf)
    order_gap = (ms[:, :K - 1] - ms[:, 1:K]).min(axis=1) if K > 1 else np.full(T, np.inf)
    info = {"group_gap": group_gap, "expert_gap": expert_gap, "order_gap": order_gap}
    return idx, gate, info


def route(x, Wr, bias, G, M, K, gk, logit_offset=None):
    return select(affinity(x, Wr, logit_offset), bias, G, M, K, gk)


def near_tie(info, tol: float = 1e-6) -> np.ndarray:
    """Tokens whose choice of groups or experts hinges on a margin below tol."""
    return (info["group_gap"] < tol) | (info["expert_gap"] < tol)
