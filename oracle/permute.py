"""Expert histogram and token permutation by expert.

The pages describe tokens being dispatched to their experts (《DeepSeek-V3
Technical Report》深度解读报告 §2.4 and §3.2) and the bias update reading the
load of every expert over the whole batch (§2.3); they fix no data layout.
Plain reading used here: rows are grouped by expert in ascending expert
order and, within an expert, by ascending token index (a stable counting
sort of the (token, slot) pairs taken in token order).
"""
from __future__ import annotations

import numpy as np


def histogram(idx, E: int) -> np.ndarray:
    """c_e = number of (token, slot) pairs routed to expert e."""
    c = np.zeros(E, dtype=np.int64)
    for e in np.asarray(idx).ravel():
        c[e] += 1
    return c.astype(np.int32)


def permute(idx, E: int):
    """Stable counting sort of routed pairs.

    Returns offsets int32 [E+1] (exclusive prefix sum of the histogram),
    sorted_token int32 [T*K] (token of each grouped row) and row_of int32
    [T][K] (grouped row of each (token, slot) pair).
    """
    idx = np.asarray(idx)
    T, K = idx.shape
    counts = histogram(idx, E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    nxt = offsets[:-1].copy()
    row_of = np.empty((T, K), dtype=np.int64)
    sorted_token = np.empty(T * K, dtype=np.int64)
    flat = idx.tolist()
    for t in range(T):
        row = flat[t]
        for k in range(K):
            e = row[k]
            r = nxt[e]
            nxt[e] = r + 1
            row_of[t, k] = r
            sorted_token[r] = t
    return offsets.astype(np.int32), sorted_token.astype(np.int32), row_of.astype(np.int32)
