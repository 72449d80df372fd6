"""Named layer shapes for the DeepSeekMoE layer forward.

The five workloads follow the DeepSeek-V3 layer as described in the
"DeepSeek-V3 Technical Report" reading notes (zako-mio knowledge base,
§2.2 DeepSeekMoE, §2.3 aux-loss-free balancing, §2.4 node-limited routing)
and the devpress blog (§1: 256 routed + 1 shared expert, 8 routed per token).

Notation: T tokens, d hidden size, E routed experts, I expert intermediate
size (the shared expert uses the same I), K routed experts per token,
G expert groups (stand-ins for nodes), M groups a token may reach, gk the
number of highest affinities summed into a group's score.
"""
from __future__ import annotations

import dataclasses
from typing import Optional


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    I: int
    K: int
    G: int
    M: int
    gk: int
    seed: int
    bias: str = "zero"              # "zero" or "uniform" (U(-0.1, 0.1))
    skew_steps: int = 0             # > 0: route + bias update loop length
    gamma: float = 1e-3             # bias update speed
    zipf_s: Optional[float] = None  # per-expert router logit offsets when set
    zipf_c: float = 0.0             # scale of those offsets
    expert_seed: Optional[int] = None  # seed of the expert weights (default: seed)

    @property
    def rows(self) -> int:
        """Rows of the grouped GEMMs: T*K routed rows followed by T shared rows."""
        return self.T * self.K + self.T

    def flops(self) -> float:
        """Algorithmic FLOPs of one layer forward (2 per multiply-add).

        Router logits 2*T*d*E, plus per (token, expert) pair and per token of
        the shared expert: gate+up projection 2*2*d*I and down projection 2*d*I.
        """
        return 2.0 * self.T * self.d * self.E + 6.0 * self.d * self.I * (self.K + 1) * self.T

    def gemm_flops(self) -> tuple[float, float]:
        """FLOPs of the two grouped FP8 GEMMs (gate/up, down)."""
        rows = self.rows
        return 4.0 * rows * self.d * self.I, 2.0 * rows * self.I * self.d

    @property
    def weight_seed(self) -> int:
        return self.seed if self.expert_seed is None else self.expert_seed

    def abi(self) -> tuple[int, ...]:
        return (self.T, self.d, self.E, self.I, self.K, self.G, self.M, self.gk)

    def with_tokens(self, T: int) -> "MoEConfig":
        return dataclasses.replace(self, T=T)


TINY = MoEConfig("tiny", T=256, d=256, E=16, I=128, K=4, G=4, M=2, gk=2, seed=0, bias="uniform")
MID = MoEConfig("mid", T=4096, d=2048, E=64, I=1408, K=6, G=8, M=3, gk=2, seed=1)
# The three full-width workloads run the same layer: one set of expert weights
# (seed 2) on different batches, routers and biases (their own seeds).
FULL = MoEConfig("full", T=16384, d=7168, E=256, I=2048, K=8, G=8, M=4, gk=2, seed=2)
DECODE = MoEConfig("decode", T=128, d=7168, E=256, I=2048, K=8, G=8, M=4, gk=2, seed=3, expert_seed=2)
# c = 0.274886: bisection with the FP64 reference router on a seeded 8192-token
# batch for a hottest-expert load of 8x the mean at step 0 (tests/golden/calibrate_skew.py)
SKEW = MoEConfig("skew", T=65536, d=7168, E=256, I=2048, K=8, G=8, M=4, gk=2, seed=4,
                 skew_steps=50, gamma=1e-3, zipf_s=1.1, zipf_c=0.274886, expert_seed=2)

CONFIGS = {c.name: c for c in (TINY, MID, FULL, DECODE, SKEW)}

# Full-width layer shapes (d, I, K, 56 K-chunks per tile) with only 32 routed
# experts and 4096 tokens: the same per-tile GEMM behaviour as the full-width
# prefill in about 3 GB of device memory, for kernel profiles.
FULLWIDTH_SMALL = MoEConfig("fullwidth_small", T=4096, d=7168, E=32, I=2048, K=8, G=8, M=4, gk=2, seed=5)
# Full-width shapes with 16 routed experts and 1024 tokens: 512 rows per expert as in the
# full-width prefill, about 4 GB of device memory for a training step, for profiles of the
# backward kernels.
FULLWIDTH_E16 = MoEConfig("fullwidth_e16", T=1024, d=7168, E=16, I=2048, K=8, G=8, M=4, gk=2, seed=6)
# The full-width prefill's token shapes (T=16384, d=7168, E=256, K=8, G=8, M=4) with an
# intermediate size of 128: the router, permutation, quantiser and combine run at exactly
# their full-width sizes (the fused router included) in about 5 GB of device memory, for
# DRAM-counter profiles of those calls.
FULLWIDTH_HBM = MoEConfig("fullwidth_hbm", T=16384, d=7168, E=256, I=128, K=8, G=8, M=4, gk=2, seed=2)
PROFILE_CONFIGS = {c.name: c for c in (FULLWIDTH_SMALL, FULLWIDTH_E16, FULLWIDTH_HBM)}
