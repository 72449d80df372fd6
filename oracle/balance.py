"""Sequence-wise balance statistics and loss L_Bal (test infrastructure, like the
rest of the oracle).

《DeepSeek-V3 Technical Report》深度解读报告 §2.3 pairs the auxiliary-loss-free bias
with a sequence-wise balance loss L_Bal of a very small weight alpha, which keeps
any single sequence from routing to a few experts. The page states only that much.
This file follows the plainest reading: the usual product of load and affinity
shares, computed per sequence.

For a sequence of L consecutive tokens t with affinities s[t][i] (sigmoid, no
bias) and chosen experts idx[t] (K of them):
  f_i = E / (K * L) * #{t : i in idx[t]}        (1 for every expert when balanced)
  P_i = (1 / L) * sum_t s[t][i] / sum_j s[t][j]  (mean normalised affinity)
  L_Bal = alpha * sum_i f_i * P_i
"""
from __future__ import annotations

import numpy as np


def balance_stats(s, idx, seq_len: int):
    """s float [T][E], idx int [T][K] -> (f, P) float64 [T/seq_len][E]."""
    s = np.asarray(s, np.float64)
    idx = np.asarray(idx)
    T, E = s.shape
    K = idx.shape[1]
    assert T % seq_len == 0
    nseq = T // seq_len
    f = np.zeros((nseq, E))
    P = np.zeros((nseq, E))
    for q in range(nseq):
        rows = slice(q * seq_len, (q + 1) * seq_len)
        counts = np.bincount(idx[rows].ravel(), minlength=E)
        f[q] = E / (K * seq_len) * counts
        P[q] = (s[rows] / s[rows].sum(axis=1, keepdims=True)).mean(axis=0)
    return f, P


def balance_loss(s, idx, seq_len: int, alpha: float) -> np.ndarray:
    """Per-sequence L_Bal, float64 [T/seq_len]."""
    f, P = balance_stats(s, idx, seq_len)
    return alpha * (f * P).sum(axis=1)
