"""Data-parallel exchange on CPU: two gloo ranks each route half of a batch
with the oracle, sum their expert loads with the package's all-reduce, and
must reach the same bias update as one process that sees the whole batch."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle.layer import bias_update
    from oracle.permute import histogram
    from oracle.route import route
    from sparse_moe_layer_13_b300 import dp, inputs
    from sparse_moe_layer_13_b300.configs import MoEConfig
    cfg = MoEConfig("dp", T=64, d=128, E=16, I=128, K=4, G=4, M=2, gk=2, seed=21, bias="uniform")
    x = inputs.gen_x(cfg).float().numpy()
    Wr = inputs.gen_router(cfg).numpy()
    b = inputs.gen_bias(cfg).numpy()
    half = cfg.T // world
    mine = x[rank * half:(rank + 1) * half]
    idx, _, _ = route(mine, Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)
    counts = torch.from_numpy(histogram(idx, cfg.E).astype(np.int32))
    dp.allreduce_load(counts)
    T_all = dp.global_tokens(half)
    nb = bias_update(b, counts.numpy(), T_all, cfg.K, cfg.gamma)
    out[rank] = torch.from_numpy(np.concatenate([counts.numpy().astype(np.float64), nb.astype(np.float64)]))
    dist.destroy_process_group()


def test_two_rank_load_allreduce_matches_single_process():
    from oracle.layer import bias_update
    from oracle.permute import histogram
    from oracle.route import route
    from sparse_moe_layer_13_b300 import inputs
    from sparse_moe_layer_13_b300.configs import MoEConfig
    world = 2
    out = torch.zeros(world, 32, dtype=torch.float64).share_memory_()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    cfg = MoEConfig("dp", T=64, d=128, E=16, I=128, K=4, G=4, M=2, gk=2, seed=21, bias="uniform")
    x = inputs.gen_x(cfg).float().numpy()
    Wr = inputs.gen_router(cfg).numpy()
    b = inputs.gen_bias(cfg).numpy()
    idx, _, _ = route(x, Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)
    c = histogram(idx, cfg.E)
    want = np.concatenate([c.astype(np.float64), bias_update(b, c, cfg.T, cfg.K, cfg.gamma).astype(np.float64)])
    for r in range(world):
        assert np.array_equal(out[r].numpy(), want)
