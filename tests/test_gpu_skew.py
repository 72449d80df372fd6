"""GPU parity of the skewed-load workload at its stated size: T = 65536 tokens
at full width, 50 steps of (route with loads -> end-of-step bias update) on
fresh batches with gamma = 1e-3, then one whole layer forward with the final
bias (《DeepSeek-V3 Technical Report》深度解读报告 §2.3 for the update; the
hottest expert's 8x start from "DeepSeek-V3的MoE架构设计革新" §6).

Every step is compared with the oracle router run from the same pre-step
bias: expert choice and gates on the tokens whose choice has a margin of at
least 1e-6, the load with near-tie tokens taken out of both histograms, and
the bias bit for bit (the update rule applied to the device's load). The
forward is compared on 64 sampled tokens, 16 of them routed to the hottest
expert. Batches are seeded as in the benchmark's balancing loop."""
import numpy as np
import torch

from gpu_helpers import (assert_y_close, check_load_and_bias, check_routing, gpu, oracle_experts,
                         oracle_route_chunked, require_gpu, to_np)
from oracle.layer import Layer
from sparse_moe_layer_13_b300.configs import SKEW


@gpu
def test_skew_balancing_loop_and_forward_match_oracle():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    cfg = SKEW
    off = inputs.gen_logit_offset(cfg, cfg.zipf_c, "cuda")
    layer = MoELayer(cfg, "cuda", logit_offset=off)
    Wr, offn = to_np(layer.Wr), to_np(off)
    mean = cfg.T * cfg.K / cfg.E
    ratios, ties = [], []
    for step in range(cfg.skew_steps):
        x = inputs.gen_x(cfg, "cuda", step=1000 + step)
        b0 = to_np(layer.bias).copy()
        binding.route(cfg, x, layer.Wr, layer.bias, off, layer.ws, layer.idx, layer.gate, layer.counts)
        binding.bias_update(cfg.E, cfg.T, cfg.K, layer.counts, cfg.gamma, layer.bias)
        binding.check_device_status()
        r_idx, r_gate, info = oracle_route_chunked(to_np(x), Wr, b0, cfg, offn)
        del x
        tie, _ = check_routing(cfg, to_np(layer.idx), to_np(layer.gate), r_idx, r_gate, info)
        check_load_and_bias(cfg, to_np(layer.idx), to_np(layer.counts), r_idx, tie, b0, to_np(layer.bias))
        ratios.append(to_np(layer.counts).max() / mean)
        ties.append(int(tie.sum()))
    print(f"[skew] max/mean load per step {np.round(ratios, 2).tolist()}; near-tie tokens per step {ties}")
    assert ratios[0] > 6.0                       # the offsets really skew the load (~8x)
    assert ratios[-1] < ratios[0]                # and the bias update pulls it down
    assert max(ties) < 0.01 * cfg.T

    # one layer forward on a fresh batch with the bias the loop left
    x = inputs.gen_x(cfg, "cuda")
    b0 = to_np(layer.bias).copy()
    y = to_np(layer.forward(x, update_bias=True))
    binding.check_device_status()
    xn = to_np(x)
    r_idx, r_gate, info = oracle_route_chunked(xn, Wr, b0, cfg, offn)
    tie, _ = check_routing(cfg, to_np(layer.idx), to_np(layer.gate), r_idx, r_gate, info)
    check_load_and_bias(cfg, to_np(layer.idx), to_np(layer.counts), r_idx, tie, b0, to_np(layer.bias))
    hot = int(np.argmax(to_np(layer.counts)))
    rng = np.random.default_rng(7)
    on_hot = np.nonzero(~tie & (r_idx == hot).any(axis=1))[0]
    hot_tok = rng.choice(on_hot, 16, replace=False)
    rest = rng.choice(np.setdiff1d(np.nonzero(~tie)[0], hot_tok), 48, replace=False)
    tokens = np.sort(np.concatenate([hot_tok, rest]))
    ex = oracle_experts(cfg, set(r_idx[tokens].ravel().tolist()) | {cfg.E})
    ref = Layer(cfg, Wr, b0, None, logit_offset=offn, experts=ex).forward(xn, tokens=tokens, idx=r_idx, gate=r_gate,
                                                                          budget=True)
    assert_y_close(y[tokens], ref["y"], ref["budget"])
    torch.cuda.synchronize()
