"""Finds the Zipf logit-offset scale c of the skewed-load workload.

The workload (hottest expert at about 8x the mean load at the first step,
"DeepSeek-V3的MoE架构设计革新" §6: early in training some hot experts carried
8x the average load) adds o_e = -c * 1.1 * ln(rank_e) to the router logits.
c is found by bisection with the FP64 oracle router on a seeded 8192-token
batch drawn on the CPU with the workload's own recipe, and written to
skew_offset.txt. Run: python tests/golden/calibrate_skew.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.permute import histogram  # noqa: E402
from oracle.route import select  # noqa: E402
from sparse_moe_layer_13_b300 import inputs  # noqa: E402
from sparse_moe_layer_13_b300.configs import SKEW  # noqa: E402

TARGET = 8.0
T_CAL = 8192


def load_ratio(z, unit_offset, c):
    cfg = SKEW
    s = 1.0 / (1.0 + np.exp(-(z + c * unit_offset[None, :])))
    idx, _, _ = select(s, np.zeros(cfg.E), cfg.G, cfg.M, cfg.K, cfg.gk)
    counts = histogram(idx, cfg.E)
    return counts.max() / (z.shape[0] * cfg.K / cfg.E)


def main():
    cfg = SKEW
    x = inputs.gen_x(cfg, "cpu", T=T_CAL).float().numpy().astype(np.float64)
    Wr = inputs.gen_router(cfg, "cpu").numpy().astype(np.float64)
    z = x @ Wr.T
    unit = inputs.gen_logit_offset(cfg, 1.0, "cpu").numpy().astype(np.float64)
    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if load_ratio(z, unit, mid) < TARGET:
            lo = mid
        else:
            hi = mid
    c = 0.5 * (lo + hi)
    r = load_ratio(z, unit, c)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "skew_offset.txt")
    with open(out, "w") as f:
        f.write("# Zipf logit-offset scale of the skewed-load workload, from calibrate_skew.py\n")
        f.write(f"# (FP64 oracle routing of a {T_CAL}-token CPU batch; max/mean load {r:.3f} at step 0)\n")
        f.write(f"c: {c:.6f}\n")
    print(c, r)


if __name__ == "__main__":
    main()
