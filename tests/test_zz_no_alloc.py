"""moe_permute_noalloc: the permutation entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

Checked through the C ABI against moe_permute, bit for bit, on two calls in
a row with different inputs, so the second call also shows that what the
first left in the shared scratch does not leak into its results. This file
sorts last so that a run stopping at the first failure has run every other
test already.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, require_gpu, to_np
from sparse_moe_layer_13_b300.configs import MoEConfig

KEYS = ("offsets", "counts", "sorted_token", "row_of", "xq_perm", "xs_perm")


def _case(cfg, seed):
    from sparse_moe_layer_13_b300 import binding, inputs
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, cfg.E + 1) ** 1.1
    idx = np.stack([rng.choice(cfg.E, cfg.K, replace=False, p=p / p.sum()) for _ in range(cfg.T)]).astype(np.int32)
    x = inputs.gen_x(cfg, "cuda", step=seed)
    xq, xs = binding.quant_1x128(x)
    return torch.from_numpy(idx).cuda(), xq, xs


@gpu
def test_noalloc_permute_matches_workspace_permute_twice():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    cfgs = [MoEConfig("a", T=3000, d=512, E=256, I=128, K=8, G=8, M=4, gk=2, seed=31),
            MoEConfig("b", T=700, d=256, E=64, I=128, K=6, G=8, M=3, gk=2, seed=32)]
    for n, cfg in enumerate(cfgs):          # two calls in a row, different shapes and inputs
        idx, xq, xs = _case(cfg, seed=40 + n)
        want = binding.permute(cfg, idx, xq, xs, want_counts=True)
        got = binding.permute_noalloc(cfg, idx, xq, xs, want_counts=True)
        binding.check_device_status()
        for k in KEYS:
            assert torch.equal(got[k], want[k]), (cfg.name, k)


@gpu
def test_noalloc_permute_rejects_shapes_beyond_its_scratch():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    # 2 * ceil(T/256) * E int32 must fit in 262144: T = 131329, E = 256 needs 262656
    cfg = MoEConfig("big", T=131329, d=128, E=256, I=128, K=1, G=8, M=4, gk=1, seed=1)
    idx = torch.zeros(cfg.T, cfg.K, dtype=torch.int32, device="cuda")
    xq = torch.zeros(cfg.T, cfg.d, dtype=torch.uint8, device="cuda")
    xs = torch.zeros(cfg.T, 1, dtype=torch.float32, device="cuda")
    out = {k: torch.zeros(1, dtype=torch.int32, device="cuda") for k in KEYS}
    with pytest.raises(binding.MoeError) as e:
        binding.permute_noalloc(cfg, idx, xq, xs, out=out)
    assert e.value.code == 2
