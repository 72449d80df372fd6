"""Data-parallel exchanges on CPU (two gloo ranks, each with half of a batch):
the expert loads summed by the package's all-reduce must give the bias update
of one process that sees the whole batch, and the weight gradients summed by
its gradient all-reduce must equal the whole batch's (the oracle's exact
float64 gradients, quantisation off)."""
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


class _GradCfg:
    T, d, E, I, K, G, M, gk, seed = 32, 128, 8, 64, 2, 4, 2, 2, 23


def _grad_case():
    """Exact oracle gradients of the seeded small layer: per-half weight gradients can be
    summed only if they are the same function of disjoint tokens."""
    from oracle.route import affinity, route
    cfg = _GradCfg()
    rng = np.random.default_rng(cfg.seed)
    x = rng.standard_normal((cfg.T, cfg.d))
    dy = rng.standard_normal((cfg.T, cfg.d))
    Wr = rng.standard_normal((cfg.E, cfg.d)) / np.sqrt(cfg.d)
    W = {e: tuple(rng.standard_normal(sh) / np.sqrt(cfg.d) for sh in ((cfg.I, cfg.d), (cfg.I, cfg.d), (cfg.d, cfg.I)))
         for e in range(cfg.E + 1)}
    idx, _, _ = route(x, Wr, np.zeros(cfg.E), cfg.G, cfg.M, cfg.K, cfg.gk)
    s_sel = np.take_along_axis(affinity(x, Wr), idx, axis=1)
    return cfg, x, dy, Wr, W, idx, s_sel


def _weight_grads(rows):
    from oracle.backward import Quantiser, layer_backward
    cfg, x, dy, Wr, W, idx, s_sel = _grad_case()
    sub = type("C", (), {"T": len(rows), "d": cfg.d, "E": cfg.E, "I": cfg.I, "K": cfg.K})()
    r = layer_backward(sub, x[rows], dy[rows], Wr, idx[rows], s_sel[rows], lambda e: W[e],
                       wgrad_experts=range(cfg.E + 1), router_experts=range(cfg.E), Q=Quantiser(on=False),
                       xd=x[rows])
    parts = [r["dWr"].get(e, np.zeros(cfg.d)) for e in range(cfg.E)]
    for e in range(cfg.E + 1):
        if e in r["dW"]:
            parts += [m.ravel() for m in r["dW"][e][:3]]
        else:                      # an expert none of these tokens chose
            parts += [np.zeros(cfg.I * cfg.d)] * 3
    return np.concatenate([np.ravel(p) for p in parts])


def _grad_rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_moe_layer_13_b300 import dp
    half = _GradCfg.T // world
    g = torch.from_numpy(_weight_grads(np.arange(rank * half, (rank + 1) * half)))
    dp.allreduce_grads([g])
    out[rank] = g
    dist.destroy_process_group()


def test_two_rank_weight_gradient_allreduce_matches_single_process():
    world = 2
    want = _weight_grads(np.arange(_GradCfg.T))
    out = torch.zeros(world, want.size, dtype=torch.float64).share_memory_()
    mp.spawn(_grad_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        np.testing.assert_allclose(out[r].numpy(), want, rtol=1e-10, atol=1e-12)


def _layer_step_rank(rank, world, port, out):
    """MoELayer.end_of_step with the data-parallel load hook, its bias-update
    call replaced by the oracle's rule on host tensors (no GPU on these ranks):
    checks which token count the layer hands to the update."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle.layer import bias_update
    from oracle.permute import histogram
    from oracle.route import route
    from sparse_moe_layer_13_b300 import dp, inputs
    from sparse_moe_layer_13_b300 import layer as layer_mod
    from sparse_moe_layer_13_b300.configs import MoEConfig
    full = MoEConfig("dp", T=64, d=128, E=16, I=128, K=4, G=4, M=2, gk=2, seed=21, bias="uniform")
    cfg = full.with_tokens(full.T // world)
    x = inputs.gen_x(full).float().numpy()
    Wr = inputs.gen_router(full).numpy()
    b = inputs.gen_bias(full).numpy()
    mine = x[rank * cfg.T:(rank + 1) * cfg.T]
    idx, _, _ = route(mine, Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)

    def host_bias_update(E, T, K, counts, gamma, bias):
        bias.copy_(torch.from_numpy(bias_update(bias.numpy(), counts.numpy(), T, K, gamma)))

    layer = object.__new__(layer_mod.MoELayer)     # no device buffers: only the end-of-step path
    layer.cfg = cfg
    layer.counts = torch.from_numpy(histogram(idx, cfg.E).astype(np.int32))
    layer.bias = torch.from_numpy(b.copy())
    real = layer_mod.B.bias_update
    layer_mod.B.bias_update = host_bias_update
    try:
        layer.end_of_step(counts_hook=dp.allreduce_load)
    finally:
        layer_mod.B.bias_update = real
    out[rank] = torch.from_numpy(np.concatenate([layer.counts.numpy().astype(np.float64),
                                                 layer.bias.numpy().astype(np.float64)]))
    dist.destroy_process_group()


def test_two_rank_layer_end_of_step_matches_single_process():
    """The layer's own end-of-step path (load all-reduce hook, then the bias
    update) on two ranks with half a batch each gives the bias of one process
    that routes the whole batch: the update must judge the summed load against
    the mean load of all ranks' tokens, not of one rank's."""
    from oracle.layer import bias_update
    from oracle.permute import histogram
    from oracle.route import route
    from sparse_moe_layer_13_b300 import inputs
    from sparse_moe_layer_13_b300.configs import MoEConfig
    world = 2
    out = torch.zeros(world, 32, dtype=torch.float64).share_memory_()
    mp.spawn(_layer_step_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    cfg = MoEConfig("dp", T=64, d=128, E=16, I=128, K=4, G=4, M=2, gk=2, seed=21, bias="uniform")
    x = inputs.gen_x(cfg).float().numpy()
    Wr = inputs.gen_router(cfg).numpy()
    b = inputs.gen_bias(cfg).numpy()
    idx, _, _ = route(x, Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)
    c = histogram(idx, cfg.E)
    nb = bias_update(b, c, cfg.T, cfg.K, cfg.gamma)
    # the half-batch mean would flip the sign for experts loaded between the two means
    assert not np.array_equal(nb, bias_update(b, c, cfg.T // world, cfg.K, cfg.gamma))
    want = np.concatenate([c.astype(np.float64), nb.astype(np.float64)])
    for r in range(world):
        assert np.array_equal(out[r].numpy(), want)
