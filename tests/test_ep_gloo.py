"""The expert-parallel step's protocol on CPU ranks (gloo, world sizes 2 and 4):
ep.EPLayer with dist_exchange, each rank owning E/R experts and routing its
own tokens, with CPU stand-ins for the device kernels built from the oracle
(FP64 expert FFNs on the E4M3 values). Every rank's output must equal the
single-process oracle layer on that rank's tokens, each token must be sent
once per destination rank and, with one expert group per rank, to at most M
ranks (《DeepSeek-V3 Technical Report》深度解读报告 §2.4)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg():
    from sparse_moe_layer_13_b300.configs import MoEConfig
    return MoEConfig("ep", T=48, d=256, E=16, I=128, K=4, G=4, M=2, gk=2, seed=27, bias="uniform")


def _row_bytes(d, K):
    return (d + 4 * (d // 128) + 8 * K + 15) // 16 * 16


class OracleKernels:
    """The expert-parallel steps on the host: routing, 1x128 quantisation and expert FFNs
    from the oracle (FP64), and the library's packed-row format written out with numpy."""

    def __init__(self, cfg, R, rank, Wr, bias, experts):
        self.cfg, self.R, self.rank = cfg, R, rank
        self.Wr, self.bias, self.experts = Wr, bias, experts

    def route_quant(self, x):
        from oracle.permute import histogram
        from oracle.quant import quant_1x128
        from oracle.route import route
        c = self.cfg
        xn = x.numpy()
        idx, gate, _ = route(xn, self.Wr, self.bias, c.G, c.M, c.K, c.gk)
        xq, xs = quant_1x128(xn)
        return (torch.from_numpy(idx), torch.from_numpy(gate.astype(np.float32)),
                torch.from_numpy(histogram(idx, c.E)), torch.from_numpy(xq), torch.from_numpy(xs))

    def dispatch(self, idx, gate, xq, xs):
        c, R = self.cfg, self.R
        n = c.E // R
        idx, gate, xq, xs = idx.numpy(), gate.numpy(), xq.numpy(), xs.numpy()
        rows = [(r, t) for r in range(R) for t in range(c.T) if (idx[t] // n == r).any()]
        send_row_of = np.full((c.T, c.K), -1, np.int32)
        for i, (r, t) in enumerate(rows):
            send_row_of[t, int(np.nonzero(idx[t] // n == r)[0][0])] = i
        rb = _row_bytes(c.d, c.K)
        buf = np.zeros((len(rows), rb), np.uint8)
        for i, (_, t) in enumerate(rows):
            packed = np.concatenate([xq[t], xs[t].astype(np.float32).view(np.uint8),
                                     idx[t].astype(np.int32).view(np.uint8), gate[t].astype(np.float32).view(np.uint8)])
            buf[i, :packed.size] = packed
        counts = np.bincount([r for r, _ in rows], minlength=R).tolist()
        return torch.from_numpy(buf), counts, torch.from_numpy(send_row_of)

    def _unpack(self, buf):
        c = self.cfg
        nk = c.d // 128
        xq = buf[:, :c.d]
        xs = np.ascontiguousarray(buf[:, c.d:c.d + 4 * nk]).view(np.float32)
        idx = np.ascontiguousarray(buf[:, c.d + 4 * nk:c.d + 4 * nk + 4 * c.K]).view(np.int32)
        gate = np.ascontiguousarray(buf[:, c.d + 4 * nk + 4 * c.K:c.d + 4 * nk + 8 * c.K]).view(np.float32)
        return xq, xs, idx, gate

    def serve(self, recv_buf):
        from oracle.ffn import expert_forward
        c = self.cfg
        n = c.E // self.R
        lo = self.rank * n
        buf = recv_buf.numpy()
        xq, xs, idx, gate = self._unpack(buf)
        out = np.zeros((buf.shape[0], c.K, c.d))
        for e in range(lo, lo + n):
            rows, slots = np.nonzero(idx == e)
            if len(rows):
                out[rows, slots] = expert_forward(xq[rows], xs[rows], self.experts[e])
        mine = (idx >= lo) & (idx < lo + n)
        partial = np.zeros((buf.shape[0], c.d))
        for k in range(c.K):                       # slot order
            partial += np.where(mine[:, k:k + 1], gate[:, k:k + 1].astype(np.float64) * out[:, k], 0.0)
        return torch.from_numpy(partial)

    def shared(self, xq, xs):
        from oracle.ffn import expert_forward
        return torch.from_numpy(expert_forward(xq.numpy(), xs.numpy(), self.experts[self.cfg.E]))

    def combine(self, shared_out, returned, send_row_of, residual=None):
        y = shared_out.numpy().copy()
        ro = send_row_of.numpy()
        ret = returned.numpy()
        for k in range(ro.shape[1]):
            has = ro[:, k] >= 0
            y[has] += ret[ro[has, k]]
        return torch.from_numpy(y)


def _setup():
    from oracle.ffn import QuantExpert
    from sparse_moe_layer_13_b300 import inputs
    cfg = _cfg()
    Wr = inputs.gen_router(cfg).numpy()
    b = inputs.gen_bias(cfg).numpy()
    experts = {e: QuantExpert(*[w.numpy() for w in inputs.gen_expert(cfg, e)]) for e in range(cfg.E + 1)}
    return cfg, Wr, b, experts


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_moe_layer_13_b300 import ep, inputs
    cfg, Wr, b, experts = _setup()
    layer = ep.EPLayer(cfg, world, rank, OracleKernels(cfg, world, rank, Wr, b, experts))
    x = inputs.gen_x(cfg, step=rank).float()
    y, st = layer.step(x, ep.dist_exchange())
    ranks = (st.send_row_of.numpy() >= 0).sum(axis=1)
    out[rank, :cfg.T * cfg.d] = y.reshape(-1)
    out[rank, cfg.T * cfg.d:cfg.T * cfg.d + cfg.T] = torch.from_numpy(ranks.astype(np.float64))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ep_protocol_on_gloo_ranks_matches_single_process(world):
    from oracle.layer import Layer
    from sparse_moe_layer_13_b300 import inputs
    cfg, Wr, b, experts = _setup()
    out = torch.zeros(world, cfg.T * cfg.d + cfg.T, dtype=torch.float64).share_memory_()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    layer = Layer(cfg, Wr, b, None, experts=experts)
    for r in range(world):
        x = inputs.gen_x(cfg, step=r).float().numpy()
        ref = layer.forward(x)
        y = out[r, :cfg.T * cfg.d].numpy().reshape(cfg.T, cfg.d)
        # the ranks' partial sums regroup the FP64 terms and carry FP32 gates
        np.testing.assert_allclose(y, ref["y"], rtol=2e-6, atol=2e-6 * np.abs(ref["y"]).max())
        ranks = out[r, cfg.T * cfg.d:].numpy()
        n = cfg.E // world
        want = np.array([len(set((ref["idx"][t] // n).tolist())) for t in range(cfg.T)])
        assert np.array_equal(ranks, want)                 # once per destination rank
        if cfg.G % world == 0:
            assert ranks.max() <= cfg.M                    # node-limited: at most M ranks
