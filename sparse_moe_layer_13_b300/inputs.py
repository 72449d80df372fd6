"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers; it contains none of the layer's
arithmetic (no quantisation, routing or FFN). Both the CUDA path and the
FP64 checker take their inputs from here, so both see the same bytes.

Recipe (all draws from ``torch.Generator`` seeded per tensor):

* x       : bf16 [T][d], N(0, 1) drawn in fp32 then rounded to bf16 (RNE).
* Wr      : fp32 [E][d], N(0, 1/d).
* bias    : fp32 [E], zeros or U(-0.1, 0.1).
* W1, W3  : fp32 [I][d] per expert, N(0, 1/d) (gate and up projections),
  seeded by the workload's expert seed (the full-width workloads share one).
* W2      : fp32 [d][I] per expert, N(0, 1/d) (down projection).
* dy      : bf16 [T][d], N(0, 1), the upstream gradient of a backward pass.
* logit offsets (skewed workload only): o_e = -c * s * ln(rank_e) with rank a
  seeded permutation of 1..E, giving a Zipf(s)-shaped expert popularity.

Expert index E is the shared expert. Values depend on the device the
generator runs on (CPU and CUDA Philox streams differ), so a check that
compares two implementations must draw once and hand the same tensors to
both.
"""
from __future__ import annotations

import math

import torch

from .configs import MoEConfig

_TAG = {"x": 1, "router": 2, "bias": 3, "w1": 4, "w3": 5, "w2": 6, "rank": 7, "dy": 8}


def _gen(cfg_seed: int, tag: str, idx: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((cfg_seed * 1_000_003 + _TAG[tag] * 65_537 + idx * 7_919) & 0x7FFF_FFFF_FFFF)
    return g


def gen_x(cfg: MoEConfig, device="cpu", step: int = 0, T: int | None = None) -> torch.Tensor:
    T = cfg.T if T is None else T
    g = _gen(cfg.seed, "x", step, device)
    return torch.randn(T, cfg.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gen_dy(cfg: MoEConfig, device="cpu", step: int = 0) -> torch.Tensor:
    g = _gen(cfg.seed, "dy", step, device)
    return torch.randn(cfg.T, cfg.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gen_router(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    g = _gen(cfg.seed, "router", 0, device)
    return torch.randn(cfg.E, cfg.d, generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(cfg.d))


def gen_bias(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    if cfg.bias == "zero":
        return torch.zeros(cfg.E, device=device, dtype=torch.float32)
    g = _gen(cfg.seed, "bias", 0, device)
    return (torch.rand(cfg.E, generator=g, device=device, dtype=torch.float32) * 0.2 - 0.1)


def gen_expert(cfg: MoEConfig, e: int, device="cpu"):
    """fp32 (W1 [I][d], W3 [I][d], W2 [d][I]) of expert e; e == E is the shared expert.
    Drawn from the workload's expert seed (cfg.weight_seed)."""
    s = 1.0 / math.sqrt(cfg.d)
    ws = cfg.weight_seed
    w1 = torch.randn(cfg.I, cfg.d, generator=_gen(ws, "w1", e, device), device=device) * s
    w3 = torch.randn(cfg.I, cfg.d, generator=_gen(ws, "w3", e, device), device=device) * s
    w2 = torch.randn(cfg.d, cfg.I, generator=_gen(ws, "w2", e, device), device=device) * s
    return w1, w3, w2


def gen_logit_offset(cfg: MoEConfig, c: float, device="cpu") -> torch.Tensor:
    """Zipf-shaped per-expert router logit offsets o_e = -c * s * ln(rank_e)."""
    g = _gen(cfg.seed, "rank", 0, "cpu")
    rank = torch.randperm(cfg.E, generator=g).to(torch.float64) + 1.0
    o = -c * float(cfg.zipf_s) * torch.log(rank)
    return o.to(torch.float32).to(device)
