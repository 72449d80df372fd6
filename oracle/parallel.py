"""Quantises oracle experts in parallel worker processes (spawned, never
forked), since the oracle's per-expert 128x128 quantisation takes seconds at
full width. Test infrastructure like the rest of the oracle."""
from __future__ import annotations

import multiprocessing as mp
import os

from .ffn import QuantExpert


def _one(job):
    e, w1, w3, w2, rule = job
    return e, QuantExpert(w1, w3, w2, rule)


def quantize_experts(jobs, max_procs: int = 32, rule: str = "fp32") -> dict:
    """jobs: iterable of (expert, W1, W3, W2) float32 arrays -> {expert: QuantExpert}."""
    jobs = [(*j, rule) for j in jobs]
    if len(jobs) <= 2:
        return dict(_one(j) for j in jobs)
    nproc = min(len(jobs), max(1, (os.cpu_count() or 2) - 1), max_procs)
    with mp.get_context("spawn").Pool(nproc) as pool:
        return dict(pool.imap_unordered(_one, jobs))
