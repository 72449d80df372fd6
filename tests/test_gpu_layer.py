"""GPU parity: the whole layer forward (route -> quant -> permute -> GEMM1
with SwiGLU -> GEMM2 -> combine -> bias update) against the FP64 oracle on
the workload shapes; at full width the oracle evaluates a seeded sample of
tokens."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_y_close, check_load_and_bias, check_routing, gpu, oracle_experts, require_gpu, to_np
from oracle.layer import Layer
from oracle.route import near_tie, route as oracle_route
from sparse_moe_layer_13_b300.configs import CONFIGS


def _layer_case(cfg, n_sample=None, residual=False, seed=0, rule="fp32"):
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    layer = MoELayer(cfg, "cuda", scale_rule=rule)
    x = inputs.gen_x(cfg, "cuda")
    b0 = to_np(layer.bias).copy()
    y = to_np(layer.forward(x, residual=residual, update_bias=True))
    binding.check_device_status()
    xn, Wr = to_np(x), to_np(layer.Wr)
    ref_idx, ref_gate, info = oracle_route(xn, Wr, b0, cfg.G, cfg.M, cfg.K, cfg.gk)
    check_routing(cfg, to_np(layer.idx), to_np(layer.gate), ref_idx, ref_gate, info)
    tie = near_tie(info)
    if n_sample is None:
        tokens = np.arange(cfg.T)
    else:
        rng = np.random.default_rng(seed)
        tokens = np.sort(rng.choice(np.nonzero(~tie)[0], n_sample, replace=False))
    needed = set(ref_idx[tokens].ravel().tolist()) | {cfg.E}
    ex = oracle_experts(cfg, needed, rule=rule)
    ref = Layer(cfg, Wr, b0, None, experts=ex, rule=rule).forward(xn, tokens=tokens, idx=ref_idx, gate=ref_gate,
                                                                  residual=residual, budget=True)
    keep = ~tie[tokens]
    rel, mx = assert_y_close(y[tokens][keep], ref["y"][keep], ref["budget"][keep])
    check_load_and_bias(cfg, to_np(layer.idx), to_np(layer.counts), ref_idx, tie, b0, to_np(layer.bias))
    return rel, mx, layer


@gpu
def test_layer_tiny():
    require_gpu()
    _layer_case(CONFIGS["tiny"])


@gpu
def test_layer_tiny_residual():
    require_gpu()
    _layer_case(CONFIGS["tiny"], residual=True)


@gpu
def test_layer_mid():
    require_gpu()
    _layer_case(CONFIGS["mid"])


@gpu
def test_layer_decode_every_token():
    require_gpu()
    _layer_case(CONFIGS["decode"])


@gpu
def test_layer_full_width_prefill_sampled():
    require_gpu()
    _layer_case(CONFIGS["full"], n_sample=64, seed=2)


@gpu
def test_layer_is_deterministic():
    require_gpu()
    from sparse_moe_layer_13_b300 import inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    cfg = CONFIGS["mid"]
    layer = MoELayer(cfg, "cuda")
    x = inputs.gen_x(cfg, "cuda")
    y1 = layer.forward(x, update_bias=False).clone()
    y2 = layer.forward(x, update_bias=False).clone()
    assert torch.equal(y1, y2)


@gpu
@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_layer_token_row_modes_agree(name):
    """Quantising straight into grouped rows, gathering a grouped copy, and
    fetching token rows by index inside the gate/up GEMM give bit-identical
    layer outputs."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    cfg = CONFIGS[name]
    layers = {"scatter": MoELayer(cfg, "cuda")}
    for mode in ("copy", "gather"):
        layers[mode] = MoELayer(cfg, "cuda", weights=layers["scatter"].w, token_rows=mode)
    x = inputs.gen_x(cfg, "cuda")
    ys = {m: L.forward(x, update_bias=False).clone() for m, L in layers.items()}
    binding.check_device_status()
    for m in ("copy", "gather"):
        assert torch.equal(ys["scatter"], ys[m]), m
        assert torch.equal(layers["scatter"].hq, layers[m].hq) and torch.equal(layers["scatter"].hs, layers[m].hs)
    assert torch.equal(layers["scatter"].xq_perm, layers["copy"].xq_perm)


@gpu
def test_layer_graph_replay_matches_eager():
    """A CUDA graph of two forwards (with the bias update) replays to the same
    outputs and bias as the same two forwards run eagerly."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    cfg = CONFIGS["tiny"]
    eager = MoELayer(cfg, "cuda")
    graphed = MoELayer(cfg, "cuda", weights=eager.w)
    x = inputs.gen_x(cfg, "cuda")
    b0 = eager.bias.clone()
    ys = []
    for _ in range(2):
        ys.append(eager.forward(x).clone())
    graphed.forward(x, update_bias=False)         # first launches outside the capture
    graphed.bias.copy_(b0)
    g = graphed.capture(x, steps=2)
    torch.cuda.synchronize()
    assert torch.equal(graphed.bias, b0)          # capturing runs nothing
    g.replay()
    torch.cuda.synchronize()
    binding.check_device_status()
    assert torch.equal(graphed.y, ys[1])
    assert torch.equal(graphed.bias, eager.bias)


@gpu
@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_layer_pow2_block_scaled(name):
    """Power-of-two scales throughout, both GEMMs on the block-scaled MMA,
    against the oracle's layer with the same scale rule."""
    require_gpu()
    _layer_case(CONFIGS[name], rule="pow2")


@gpu
def test_layer_pow2_block_scaled_full_width_sampled():
    require_gpu()
    _layer_case(CONFIGS["full"], n_sample=48, seed=5, rule="pow2")
