"""Expert parallelism with node-limited routing, on top of the C-ABI calls.

《DeepSeek-V3 Technical Report》深度解读报告 §2.4 limits each token to at most
M nodes (chosen by the sum of their experts' highest affinities) so that the
cross-node traffic of expert parallelism stays bounded, and §3.2 sends
tokens between nodes by all-to-all with the experts spread over the GPUs.
Here R ranks split the E routed experts into contiguous ranges of E/R (with
R dividing G a rank holds whole expert groups, the groups standing in for
nodes, so a token reaches at most M ranks); every rank holds the router and
the shared expert and routes its own T tokens. One step:

  begin   route (with loads), quantise the tokens per 1x128 tile, and pack
          each token once per destination rank (moe_ep_dispatch)
  --      all-to-all of the packed rows (split sizes: rows per rank)
  serve   group the received pairs by local expert (moe_ep_receive), run the
          two grouped FP8 GEMMs over the local experts, and sum each
          received row's gate-weighted expert outputs (moe_ep_partial)
  --      the reverse all-to-all of the partial rows, in received order,
          which brings them back in send order
  finish  the shared expert on the rank's own tokens, then y = shared +
          returned partials (moe_ep_combine)

The steps go through a `kernels` object: DeviceKernels (the library on the
GPU) by default; anything with the same methods works, so the protocol
itself can run on CPU ranks. The exchange is a callable (buf, counts) ->
(received, received counts): dist_exchange for torch.distributed ranks, or
emulate() for R ranks in one process.
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist

from . import binding as B


@dataclasses.dataclass
class SendState:
    """What a rank keeps between begin() and finish()."""
    x: torch.Tensor
    idx: torch.Tensor
    gate: torch.Tensor
    counts: torch.Tensor          # this rank's expert load (for the bias update)
    xq: torch.Tensor
    xs: torch.Tensor
    send_buf: torch.Tensor        # [S][row bytes]
    send_counts: list             # rows for each rank
    send_row_of: torch.Tensor     # [T][K] send row of each (token, first slot on a rank), else -1


class DeviceKernels:
    """The expert-parallel steps on the GPU through the library. `weights` holds every
    expert (an ExpertWeights); rank r uses the slice of experts it owns and the shared one."""

    def __init__(self, cfg, R: int, rank: int, Wr: torch.Tensor, bias: torch.Tensor, weights,
                 logit_offset: torch.Tensor | None = None):
        if cfg.E % R or not 0 <= rank < R:
            raise ValueError(f"{R} ranks do not split {cfg.E} experts evenly, or rank {rank} is out of range")
        self.cfg, self.R, self.rank = cfg, R, rank
        n = cfg.E // R
        lo = rank * n
        self.q13, self.s13 = weights.q13[lo:lo + n], weights.s13[lo:lo + n]
        self.q2, self.s2 = weights.q2[lo:lo + n], weights.s2[lo:lo + n]
        E = cfg.E
        self.sq13, self.ss13 = weights.q13[E:E + 1], weights.s13[E:E + 1]
        self.sq2, self.ss2 = weights.q2[E:E + 1], weights.s2[E:E + 1]
        self.planes = B.router_planes(Wr)
        self.bias = bias
        self.logit_offset = logit_offset
        dev = Wr.device
        self.ws = torch.empty(B.workspace_size(cfg), dtype=torch.uint8, device=dev)
        self.shared_offsets = torch.tensor([0, cfg.T], dtype=torch.int32, device=dev)

    def route_quant(self, x):
        c = self.cfg
        idx, gate, counts = B.route_planes(c, x, self.planes, self.bias, self.logit_offset, self.ws, want_counts=True)
        xq, xs = B.quant_1x128(x)
        return idx, gate, counts, xq, xs

    def dispatch(self, idx, gate, xq, xs):
        d = B.ep_dispatch(self.cfg, self.R, idx, gate, xq, xs)
        counts = d["send_counts"].tolist()               # the all-to-all needs the split sizes on the host
        return d["send_buf"][:sum(counts)], counts, d["send_row_of"]

    def serve(self, recv_buf):
        c = self.cfg
        n = recv_buf.shape[0]
        if n == 0:
            return torch.empty(0, c.d, dtype=torch.float32, device=recv_buf.device)
        r = B.ep_receive(c, self.R, self.rank, recv_buf)
        off = r["local_offsets"]
        hq, hs = B.grouped_gemm_fp8(off, r["xq_local"], r["xs_local"], self.q13, self.s13, B.MOE_EPI_SWIGLU_FP8)
        out, _ = B.grouped_gemm_fp8(off, hq, hs, self.q2, self.s2, B.MOE_EPI_BF16)
        return B.ep_partial(c, recv_buf, r["row_of"], out)

    def shared(self, xq, xs):
        hq, hs = B.grouped_gemm_fp8(self.shared_offsets, xq, xs, self.sq13, self.ss13, B.MOE_EPI_SWIGLU_FP8)
        out, _ = B.grouped_gemm_fp8(self.shared_offsets, hq, hs, self.sq2, self.ss2, B.MOE_EPI_F32)
        return out

    def combine(self, shared_out, returned, send_row_of, residual=None):
        return B.ep_combine(self.cfg, shared_out, returned, send_row_of, residual)


class EPLayer:
    """One rank of the expert-parallel layer."""

    def __init__(self, cfg, R: int, rank: int, kernels):
        self.cfg, self.R, self.rank, self.k = cfg, R, rank, kernels

    def begin(self, x) -> SendState:
        idx, gate, counts, xq, xs = self.k.route_quant(x)
        buf, send_counts, row_of = self.k.dispatch(idx, gate, xq, xs)
        return SendState(x, idx, gate, counts, xq, xs, buf, send_counts, row_of)

    def serve(self, recv_buf):
        return self.k.serve(recv_buf)

    def finish(self, st: SendState, returned, residual: bool = False):
        if returned.shape[0] != st.send_buf.shape[0]:
            raise RuntimeError(f"{returned.shape[0]} partial rows came back for {st.send_buf.shape[0]} sent")
        shared = self.k.shared(st.xq, st.xs)
        return self.k.combine(shared, returned, st.send_row_of, st.x if residual else None)

    def step(self, x, exchange, residual: bool = False):
        """One forward with a real exchange (e.g. dist_exchange()); returns (y, state)."""
        st = self.begin(x)
        recv, recv_counts = exchange(st.send_buf, st.send_counts)
        partial = self.serve(recv)
        returned, _ = exchange(partial, recv_counts)
        return self.finish(st, returned, residual), st


def dist_exchange(group=None):
    """All-to-all over torch.distributed ranks (NCCL for device tensors, gloo for host ones):
    rows [sum(counts)][...] split by `counts` (rows for each rank, in rank order) ->
    (received rows concatenated in source-rank order, rows from each rank)."""

    def exchange(buf, counts):
        sc = torch.tensor(counts, dtype=torch.int64, device=buf.device)
        rc = torch.empty_like(sc)
        dist.all_to_all_single(rc, sc, group=group)
        recv_counts = rc.tolist()
        out = buf.new_empty((sum(recv_counts),) + tuple(buf.shape[1:]))
        dist.all_to_all_single(out, buf.contiguous(), output_split_sizes=recv_counts, input_split_sizes=list(counts),
                               group=group)
        return out, recv_counts

    return exchange


def _local_all_to_all(bufs, counts):
    """bufs[s] rows for every rank r in order, counts[s][r] of them -> per r: rows from every s."""
    R = len(bufs)
    starts = [[sum(counts[s][:r]) for r in range(R + 1)] for s in range(R)]
    recv = [torch.cat([bufs[s][starts[s][r]:starts[s][r + 1]] for s in range(R)]) for r in range(R)]
    recv_counts = [[counts[s][r] for s in range(R)] for r in range(R)]
    return recv, recv_counts


def emulate(layers, xs, residual: bool = False):
    """R ranks in one process: every phase runs each rank's kernels in turn, and the two
    all-to-alls are copies between the ranks' buffers made between phases (no kernel ever
    waits on another rank's). Returns (per-rank y, per-rank SendState)."""
    states = [L.begin(x) for L, x in zip(layers, xs)]
    recv, recv_counts = _local_all_to_all([s.send_buf for s in states], [s.send_counts for s in states])
    partials = [L.serve(r) for L, r in zip(layers, recv)]
    returned, _ = _local_all_to_all(partials, recv_counts)
    return [L.finish(s, ret, residual) for L, s, ret in zip(layers, states, returned)], states
