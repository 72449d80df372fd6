"""Data-parallel replicas of the layer: the only exchange on the path.

Every step except the bias update is independent per token, so each rank
runs the whole layer on its own tokens. The end-of-step bias update reads
the load of every expert over the whole batch (《DeepSeek-V3 Technical
Report》深度解读报告 §2.3), so the per-expert counts are summed over ranks
before it, and the mean load uses the global token count.

A training step adds one more exchange: the gradients of the weights (the
router's and every expert's) are sums over tokens, so replicas that ran the
backward on disjoint tokens add theirs (allreduce_grads). The input
gradient stays with its rank.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def world(group=None) -> int:
    return dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1


def allreduce_load(counts: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the int32 per-expert load over the data-parallel ranks, in place."""
    if world(group) > 1:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return counts


def global_tokens(T_local: int, group=None) -> int:
    """Tokens of the whole data-parallel batch (every rank holds T_local)."""
    return T_local * world(group)


def allreduce_grads(grads, group=None):
    """Sums weight-gradient tensors (e.g. MoELayer.backward's dWr, dW13, dW2T) over the
    data-parallel ranks, in place; returns them. With FP8 weight gradients each rank's
    128-token tiles cover its own rows of an expert, so the sum equals one process's
    gradient up to the quantisation of differently cut tiles."""
    if world(group) > 1:
        for g in grads:
            dist.all_reduce(g, op=dist.ReduceOp.SUM, group=group)
    return grads
