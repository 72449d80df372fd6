"""GPU parity of the aux-loss-free balancing loop on the skewed workload:
steps of (route with counts -> end-of-step bias update) on fresh batches,
compared with the oracle step by step (bias bit for bit, loads exact), at
full width with a reduced token count. The inputs are seeded, so a choice
that hinges on a margin below the GPU's rounding would fail every run, not
intermittently."""
import numpy as np
import torch

from gpu_helpers import gpu, require_gpu, to_np
from oracle.layer import bias_update
from oracle.permute import histogram
from oracle.route import route as oracle_route
from sparse_moe_layer_13_b300.configs import SKEW


@gpu
def test_skew_balancing_loop_matches_oracle():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    cfg = SKEW.with_tokens(2048)
    off = inputs.gen_logit_offset(cfg, cfg.zipf_c, "cuda")
    Wr = inputs.gen_router(cfg, "cuda")
    bias = inputs.gen_bias(cfg, "cuda")
    ref_b = to_np(bias).copy()
    ws = torch.empty(binding.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    ratios = []
    for step in range(6):
        x = inputs.gen_x(cfg, "cuda", step=step)
        idx, gate, counts = binding.route(cfg, x, Wr, bias, off, ws, want_counts=True)
        binding.bias_update(cfg.E, cfg.T, cfg.K, counts, cfg.gamma, bias)
        binding.check_device_status()
        r_idx, r_gate, info = oracle_route(to_np(x), to_np(Wr), ref_b, cfg.G, cfg.M, cfg.K, cfg.gk, to_np(off))
        r_counts = histogram(r_idx, cfg.E)
        assert np.array_equal(to_np(counts), r_counts)
        ref_b = bias_update(ref_b, r_counts, cfg.T, cfg.K, cfg.gamma)
        assert np.array_equal(to_np(bias), ref_b)
        ratios.append(r_counts.max() / (cfg.T * cfg.K / cfg.E))
    assert ratios[0] > 4.0            # the offsets really skew the load
