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


def _stored_logits(cfg, ws):
    """The logits the router left in the workspace: (split count word, summed logits [T][E]),
    the K-split partials summed in split order in FP32 as the kernels add them."""
    raw = ws.cpu().numpy()
    splits = int(raw[:4].view(np.int32)[0])
    z = raw[256:256 + splits * cfg.T * cfg.E * 4].view(np.float32).reshape(splits, cfg.T, cfg.E)
    acc = z[0].copy()
    for s in range(1, splits):
        acc = (acc + z[s]).astype(np.float32)
    return splits, acc


@gpu
@pytest.mark.parametrize("T", [16384, 16384 + 37])
def test_route_fused_equals_split_path_bit_for_bit(T):
    """At full width the token tiles alone fill the SMs, so the sliced path runs one K slice
    per tile: its stored sums must equal the fused kernel's bit for bit, and so must the
    choice, gates and loads."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    cfg = CONFIGS["full"].with_tokens(T)
    x = inputs.gen_x(cfg, "cuda")
    Wr = inputs.gen_router(cfg, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    bias = (torch.rand(cfg.E, generator=g, device="cuda") - 0.5) * 0.02
    planes = binding.router_planes(Wr)
    out = {}
    for path in ("split", "fused"):
        ws = torch.zeros(binding.workspace_size(cfg), dtype=torch.uint8, device="cuda")
        idx, gate, counts = binding.route_planes(cfg, x, planes, bias, workspace=ws, want_counts=True, path=path)
        binding.check_device_status()
        out[path] = (idx, gate, counts, *_stored_logits(cfg, ws))
    assert out["split"][3] == 1 and out["fused"][3] == 1
    assert np.array_equal(out["split"][4], out["fused"][4])
    for i in range(3):
        assert torch.equal(out["split"][i], out["fused"][i])


@gpu
@pytest.mark.parametrize("name,T", [("tiny", None), ("tiny", 300), ("mid", None), ("mid", 1)])
def test_route_fused_path_matches_oracle(name, T):
    """The fused router forced on shapes where the automatic choice takes the split path
    (few token tiles, E = 16 and 64, a ragged tail, a single token)."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    c = CONFIGS[name] if T is None else CONFIGS[name].with_tokens(T)
    x = inputs.gen_x(c, "cuda")
    Wr = inputs.gen_router(c, "cuda")
    b = inputs.gen_bias(c, "cuda")
    idx, gate, counts = binding.route_planes(c, x, binding.router_planes(Wr), b, want_counts=True, path="fused")
    binding.check_device_status()
    ref_idx, ref_gate, info = oracle_route(to_np(x), to_np(Wr), to_np(b), c.G, c.M, c.K, c.gk)
    check_routing(c, to_np(idx), to_np(gate), ref_idx, ref_gate, info)
    assert np.array_equal(to_np(counts), histogram(to_np(idx), c.E))


@gpu
def test_route_fused_all_experts_one_group():
    """Fused path on the degenerate selections: K = E (every expert chosen) and G = 1."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    for c in (MoEConfig("allk", T=200, d=256, E=16, I=128, K=16, G=2, M=2, gk=1, seed=9, bias="uniform"),
              MoEConfig("g1", T=130, d=128, E=32, I=128, K=5, G=1, M=1, gk=3, seed=10, bias="uniform")):
        x = inputs.gen_x(c, "cuda")
        Wr = inputs.gen_router(c, "cuda")
        b = inputs.gen_bias(c, "cuda")
        idx, gate, _ = binding.route_planes(c, x, binding.router_planes(Wr), b, path="fused")
        binding.check_device_status()
        ref_idx, ref_gate, info = oracle_route(to_np(x), to_np(Wr), to_np(b), c.G, c.M, c.K, c.gk)
        check_routing(c, to_np(idx), to_np(gate), ref_idx, ref_gate, info)


@gpu
def test_route_planes_rejects_fused_beyond_256_experts():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    c = MoEConfig("e512", T=64, d=128, E=512, I=128, K=8, G=8, M=4, gk=2, seed=12)
    x = inputs.gen_x(c, "cuda")
    Wr = inputs.gen_router(c, "cuda")
    with pytest.raises(binding.MoeError) as e:
        binding.route_planes(c, x, binding.router_planes(Wr), torch.zeros(c.E, device="cuda"), path="fused")
    assert e.value.code == 2


@gpu
def test_route_experts_beyond_one_tile_ragged():
    """E = 320: two expert tiles of the sliced logits kernel, the last one 64 wide (its
    weight box still carries 256 rows), with a ragged token tail."""
    require_gpu()
    _run(MoEConfig("e320", T=300, d=256, E=320, I=128, K=8, G=4, M=2, gk=2, seed=13, bias="uniform"))


@gpu
@pytest.mark.parametrize("name", ["full", "decode"])
def test_router_logits_within_stated_bound(name):
    """Pins the router bound the oracle's gate error rests on (oracle/bounds.py,
    ROUTER_LOGIT_ERR): the logits the router leaves in the workspace (fused path at full
    width, sliced path for the decode batch) lie within it of x . Wr in FP64."""
    require_gpu()
    from oracle.bounds import ROUTER_LOGIT_ERR
    from sparse_moe_layer_13_b300 import binding, inputs
    cfg = CONFIGS[name]
    x = inputs.gen_x(cfg, "cuda")
    Wr = inputs.gen_router(cfg, "cuda")
    ws = torch.zeros(binding.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    binding.route(cfg, x, Wr, inputs.gen_bias(cfg, "cuda"), None, ws)
    binding.check_device_status()
    _, z = _stored_logits(cfg, ws)
    tok = np.arange(0, cfg.T, 7)
    exact = to_np(x)[tok].astype(np.float64) @ to_np(Wr).astype(np.float64).T
    err = np.abs(z[tok].astype(np.float64) - exact)
    print(f"[router] {name}: max |logit - exact| {err.max():.3e}, mean {err.mean():.3e} (bound {ROUTER_LOGIT_ERR:g})")
    assert err.max() <= ROUTER_LOGIT_ERR
