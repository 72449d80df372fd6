"""GPU parity: router (affinity, group-limited aux-loss-free top-K, gates,
histogram) against the oracle on the workload shapes."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_routing, gpu, require_gpu, to_np
from oracle.permute import histogram
from oracle.route import route as oracle_route
from sparse_moe_layer_13_b300.configs import CONFIGS, MoEConfig


def _run(cfg, T=None, logit_offset=None, bias=None):
    from sparse_moe_layer_13_b300 import binding, inputs
    c = cfg if T is None else cfg.with_tokens(T)
    x = inputs.gen_x(c, "cuda")
    Wr = inputs.gen_router(c, "cuda")
    b = inputs.gen_bias(c, "cuda") if bias is None else bias
    idx, gate, counts = binding.route(c, x, Wr, b, logit_offset, want_counts=True)
    binding.check_device_status()
    ref_idx, ref_gate, info = oracle_route(to_np(x), to_np(Wr), to_np(b), c.G, c.M, c.K, c.gk,
                                           None if logit_offset is None else to_np(logit_offset))
    tie, err = check_routing(c, to_np(idx), to_np(gate), ref_idx, ref_gate, info)
    # histogram of the device's own choice, bit-exact
    assert np.array_equal(to_np(counts), histogram(to_np(idx), c.E))
    assert tie.mean() < 0.01
    return err


@gpu
@pytest.mark.parametrize("name", ["tiny", "mid", "full", "decode"])
def test_route_workloads(name):
    require_gpu()
    _run(CONFIGS[name])


@gpu
@pytest.mark.parametrize("T", [1, 3, 300])
def test_route_ragged_token_counts(T):
    require_gpu()
    _run(CONFIGS["tiny"], T=T)
    _run(CONFIGS["mid"], T=T)


@gpu
def test_route_biased_selection_and_offsets():
    require_gpu()
    cfg = CONFIGS["mid"].with_tokens(2048)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    bias = (torch.rand(cfg.E, generator=g, device="cuda") - 0.5) * 0.2
    off = torch.randn(cfg.E, generator=g, device="cuda")
    _run(cfg, bias=bias, logit_offset=off)


@gpu
def test_route_all_groups_all_experts():
    require_gpu()
    cfg = MoEConfig("allk", T=64, d=256, E=16, I=128, K=16, G=2, M=2, gk=1, seed=9, bias="uniform")
    _run(cfg)
    cfg = MoEConfig("g1", T=100, d=128, E=32, I=128, K=5, G=1, M=1, gk=3, seed=10, bias="uniform")
    _run(cfg)


@gpu
@pytest.mark.parametrize("name,seq_len", [("tiny", 64), ("mid", 1024), ("full", 4096)])
def test_balance_loss_matches_oracle(name, seq_len):
    """Sequence-wise balance statistics from the router's own logits against
    the oracle's FP64 affinities and the GPU's routing."""
    require_gpu()
    from oracle.balance import balance_stats
    from oracle.route import affinity
    from sparse_moe_layer_13_b300 import binding, inputs
    cfg = CONFIGS[name]
    x = inputs.gen_x(cfg, "cuda")
    Wr = inputs.gen_router(cfg, "cuda")
    bias = inputs.gen_bias(cfg, "cuda")
    ws = torch.empty(binding.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx, gate, _ = binding.route(cfg, x, Wr, bias, None, ws)
    loss, f, P = binding.balance_loss(cfg, idx, ws, seq_len, 1e-4)
    binding.check_device_status()
    s = affinity(to_np(x), to_np(Wr))
    rf, rP = balance_stats(s, to_np(idx), seq_len)
    assert np.allclose(to_np(f), rf, rtol=1e-6, atol=0)          # counts exact; E / (K L) rounded in FP32
    assert np.allclose(to_np(P), rP, rtol=1e-5, atol=1e-9)
    assert np.allclose(to_np(loss), 1e-4 * (rf * rP).sum(axis=1), rtol=1e-5, atol=0)
