"""Benchmark: DeepSeekMoE layer forward on B300, one JSON line on stdout.

Workload: the full-width prefill layer (T=16384 tokens, d=7168, 256 routed +
1 shared SwiGLU experts, I=2048, top-8, 8 groups / at most 4 per token),
synthetic seeded inputs and random-init weights. A step is one whole layer
forward: route -> permute -> quantise into grouped rows -> grouped FP8 GEMM
(gate/up, SwiGLU, requantise) -> grouped FP8 GEMM (down) -> combine -> bias
update.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config full]
  python bench.py --impl reference ...   # the FP64 CPU oracle on a token sample
  python bench.py --backward ...         # a training step: forward, bias update, backward

Under torchrun (N > 1) each rank runs its own layer on its own tokens (weak
scaling); the only exchange is an all-reduce of the per-expert load before
the bias update. value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# measured DRAM bytes / algorithmic bytes of the gate/up GEMM (ncu, fullwidth_small workload,
# the current kernel: 1.490 GB against 1.319 GB)
GATE_UP_DRAM_OVER_ALGORITHMIC = 1.129
METRIC = "MoE layer tokens/s; FP8 grouped-GEMM TFLOP/s & % of roofline (1 B300)"
UNIT = "tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), d.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def _fp8_peak(bf16, bf16_s, src, clock_summary):
    """FP8 dense peak (2 x bf16, the nominal E4M3 : bf16 ratio) for a contraction timed inside
    the run of K back-to-back steps: the sustained (power-capped) bf16 figure when the clock
    record of the timed region shows the power cap active, else the burst figure."""
    capped = bf16_s is not None and "sw_power_cap" in (clock_summary.get("reasons") or [])
    b = bf16_s if capped else bf16
    kind = "sustained, power cap active in the timed region" if capped else "burst"
    return 2.0 * b, f"{src}: bf16 {kind} {b} TFLOP/s x 2 (E4M3/bf16 nominal ratio)"


def time_alone(fn, reps: int = 10, pause_s: float = 0.05) -> float:
    """Best of `reps` single launches of fn (ms, CUDA events on the current stream), each
    after a pause with the GPU idle: the regime of the measured peaks' burst figures (best
    of 10 short runs), as against the power-capped run of K back-to-back steps."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        time.sleep(pause_s)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return best


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from sparse_moe_layer_13_b300 import binding, dp, inputs
    from sparse_moe_layer_13_b300.configs import CONFIGS, PROFILE_CONFIGS
    from sparse_moe_layer_13_b300.layer import MoELayer

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if ws > 1:
        dist.barrier()
    cfg = {**CONFIGS, **PROFILE_CONFIGS}[args.config]
    offset = inputs.gen_logit_offset(cfg, cfg.zipf_c, dev) if cfg.zipf_s else None
    layer = MoELayer(cfg, dev, logit_offset=offset, scale_rule=args.scales)
    skew = None
    if cfg.skew_steps:
        skew = balancing_loop(cfg, layer, dev, binding, inputs, dp)
    # each rank its own tokens: a different x batch per rank
    x = inputs.gen_x(cfg, dev, step=rank)
    hook = dp.allreduce_load if ws > 1 else None
    # the bias update judges the load of the whole data-parallel batch
    T_all = dp.global_tokens(cfg.T)

    def _step(events=None):
        y = layer.forward(x, update_bias=False, events=events)
        if hook is not None:
            hook(layer.counts)
        binding.bias_update(cfg.E, T_all, cfg.K, layer.counts, cfg.gamma, layer.bias)
        return y

    for _ in range(args.warmup):
        _step()
    torch.cuda.synchronize()
    binding.check_device_status()

    K = args.steps
    # GEMM events are external so that, inside a CUDA graph, they become real event records
    calls = ("route", "permute", "quant", "gemm1", "gemm2", "combine")
    ev = {n: [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
              for _ in range(K)] for n in calls}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # one GPU: the K timed steps run as one CUDA graph (13 launches per step, no host work
    # between them); it is replayed once untimed first. Under torchrun the steps run eagerly.
    graph = None
    if ws == 1 and not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(K):
                _step({n: ev[n][i] for n in ev})
        graph.replay()
        torch.cuda.synchronize()
        binding.check_device_status()
    with ClockSampler(local) as clocks:
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record()
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                _step({n: ev[n][i] for n in ev})
        t1.record()
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
    binding.check_device_status()
    ms = t0.elapsed_time(t1) / K
    kt = {n: statistics.mean(a.elapsed_time(b) for a, b in ev[n]) for n in calls}
    if ws > 1:
        t = torch.tensor([ms] + [kt[n] for n in calls], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, *rest = t.tolist()
        kt = dict(zip(calls, rest))
    g1, g2 = kt["gemm1"], kt["gemm2"]

    # End to end through the public API: every step copies its x from pinned host
    # memory and its y back to pinned host memory. Copies run on their own streams
    # and overlap the neighbouring steps' compute (x and y double-buffered).
    e2e_ms = e2e_pipelined(cfg, layer, x, K, hook, binding, T_all)
    if ws > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = t.item()
    # the gate/up GEMM alone on the last step's grouped rows, best of 10 single launches
    g1_alone = None
    if ws == 1 and not args.eager:
        def _gate_up():
            binding.grouped_gemm_fp8(layer.perm["offsets"], layer.xq_perm, layer.xs_perm, layer.w.q13, layer.w.s13,
                                     binding.MOE_EPI_SWIGLU_FP8, layer.hq, layer.hs,
                                     block_scaled=layer.block_scaled)
        g1_alone = time_alone(_gate_up)
        binding.check_device_status()

    hbm, bf16, bf16_s, src = _peaks()
    f1, f2 = cfg.gemm_flops()
    fp8_peak = 2.0 * bf16          # E4M3 dense rate is twice bf16 (4.5 vs 2.25 PFLOP/s nominal)
    clock_summary = clocks.summary()
    roof_peak, roof_src = _fp8_peak(bf16, bf16_s, src, clock_summary)
    g1_tflops = f1 / (g1 * 1e-3) / 1e12
    g2_tflops = f2 / (g2 * 1e-3) / 1e12
    # weight bytes the gate/up GEMM must stream: every expert that received a token, plus the shared one
    touched = int((layer.counts > 0).sum().item()) + 1
    w13_bytes = touched * (2 * cfg.I * cfg.d + 4 * (2 * cfg.I // 128) * (cfg.d // 128))
    a_bytes = cfg.rows * (cfg.d + 4 * cfg.d // 128) + cfg.rows * (cfg.I + 4 * cfg.I // 128)
    g1_gbs = (w13_bytes + a_bytes) / (g1 * 1e-3) / 1e9
    # DRAM bytes per gate/up launch: ncu's dram__bytes_read.sum + dram__bytes_write.sum for the
    # same kernel on the fullwidth_small workload (small enough to capture) were 1.129 x its
    # algorithmic bytes; traffic grows with the touched weights and rows, so a launch of this
    # workload is estimated at that ratio.
    traffic = round(GATE_UP_DRAM_OVER_ALGORITHMIC * (w13_bytes + a_bytes))
    weight_bound = cfg.T <= 1024     # a few rows per expert: the GEMMs stream weights
    if weight_bound:
        roof = {"kernel": "grouped_gemm_fp8 gate/up + SwiGLU (streams the touched experts' W13)",
                "bound": "hbm", "achieved": round(g1_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(g1_gbs / hbm, 4), "traffic": None,
                "algorithmic_bytes": w13_bytes + a_bytes, "touched_experts": touched,
                "peak_source": f"{src}: HBM copy bandwidth"}
    else:
        roof = {"kernel": "grouped_gemm_fp8 gate/up + SwiGLU (largest share of the step)",
                "bound": "tensor", "achieved": round(g1_tflops, 1), "peak": round(roof_peak, 1),
                "unit": "TFLOP/s", "frac": round(g1_tflops / roof_peak, 4),
                "frac_of_burst": round(g1_tflops / fp8_peak, 4), "traffic": traffic,
                "traffic_note": "DRAM bytes per launch, scaled from an ncu capture of the fullwidth_small workload",
                "algorithmic_bytes": w13_bytes + a_bytes, "peak_source": roof_src}
    tokens = cfg.T * ws
    value = tokens / (ms * 1e-3)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic (seeded N(0,1) x, N(0,1/d) weights, random init)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E}+1 I={cfg.I} K={cfg.K} G={cfg.G} M={cfg.M}"
                               + (" (power-of-two scales, block-scaled GEMMs)" if args.scales == "pow2" else ""),
                   "scale_rule": args.scales,
                   "tokens_per_gpu": cfg.T, "global_tokens": tokens, "parallelism": f"dp{ws}",
                   "launch": "one CUDA graph of the K steps" if graph is not None else "eager launches",
                   "l2": (f"inputs exceed L2: x {cfg.T * cfg.d * 2 / 1e6:.0f} MB and FP8 expert weights "
                          f"{(cfg.E + 1) * 3 * cfg.d * cfg.I / 1e9:.2f} GB read every step, no flush")},
        "layer_tflops": round(cfg.flops() * ws / (ms * 1e-3) / 1e12, 1),
        "gemm": {"gate_up_swiglu_ms": round(g1, 4), "gate_up_tflops": round(g1_tflops, 1),
                 "down_ms": round(g2, 4), "down_tflops": round(g2_tflops, 1),
                 "grouped_gemm_tflops": round((f1 + f2) / ((g1 + g2) * 1e-3) / 1e12, 1),
                 "gate_up_gbs": round(g1_gbs, 1),
                 "gate_up_alone": None if g1_alone is None else {
                     "ms": round(g1_alone, 4), "tflops": round(f1 / (g1_alone * 1e-3) / 1e12, 1),
                     "frac_of_burst": round(f1 / (g1_alone * 1e-3) / 1e12 / fp8_peak, 4),
                     "how": "best of 10 single launches 50 ms apart on the last step's grouped rows, "
                            "against 2 x the bf16 burst figure (cuBLAS best of 10)"}},
        "roofline": roof,
        "kernels": call_table(cfg, kt, w13_bytes + a_bytes, hbm, bf16, fp8_peak, layer.route_fused),
        "e2e": {"value": round(tokens / (e2e_ms * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2},
        "gpu_launches": K * layer.launches_per_forward,
        **({"skew": skew} if skew else {}),
        "clocks": clock_summary,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, n_tokens=args.cpu_tokens, steps=1)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def call_table(cfg, kt, gemm1_bytes, hbm, bf16, fp8_peak, fused):
    """Per-call device time (CUDA events around each call inside the timed step, mean over
    the K steps), algorithmic bytes and FLOPs, and the fractions of the measured HBM copy
    bandwidth and tensor peaks they reach. Algorithmic bytes count each input read once and
    each output written once:
      route    x T*d*2 + weight planes 3*E*d*2 + choice and gates T*K*8 + summed logits
               T*E*4 (kept for the backward pass) + the load histogram's read T*K*4;
               FLOPs 3 * 2*T*d*E (x times the three bf16 terms of Wr, bf16 tensor cores)
      permute  choice T*K*4 read; grouped row lists (T*K+T)*4 and row_of T*K*4 written
      quant    x T*d*2 and row_of T*K*4 read; E4M3 rows R*d and scales R*d/128*4 written
      gemm1    touched W13 and scales, grouped x rows and scales, h and its scales
      gemm2    FLOPs 2*R*I*d (its bytes are dominated by the same weight stream)
      combine  routed rows T*K*d*2 (bf16) + shared rows T*d*4 (FP32) + row_of and gates
               T*K*8 read; y T*d*2 written
    with R = T*K + T grouped rows."""
    T, d, E, I, K = cfg.T, cfg.d, cfg.E, cfg.I, cfg.K
    R = T * K + T
    f1, f2 = cfg.gemm_flops()
    work = {
        "route": (T * d * 2 + 3 * E * d * 2 + T * K * 8 + T * E * 4 + T * K * 4, 6.0 * T * d * E, bf16),
        "permute": (T * K * 4 + R * 4 + T * K * 4, None, None),
        "quant": (T * d * 2 + T * K * 4 + R * d + R * (d // 128) * 4, None, None),
        "gemm1": (gemm1_bytes, f1, fp8_peak),
        "gemm2": (None, f2, fp8_peak),
        "combine": (T * K * d * 2 + T * d * 4 + T * K * 8 + T * d * 2, None, None),
    }
    out = {}
    for n, (nbytes, flops, peak) in work.items():
        ms = kt.get(n)
        if not ms:
            continue
        e = {"ms": round(ms, 4)}
        if nbytes is not None:
            gbs = nbytes / (ms * 1e-3) / 1e9
            e.update(bytes=int(nbytes), gbs=round(gbs, 1), hbm_frac=round(gbs / hbm, 4))
        if flops is not None:
            tf = flops / (ms * 1e-3) / 1e12
            e.update(tflops=round(tf, 1), tensor_frac=round(tf / peak, 4))
        out[n] = e
    out["route"]["path"] = "fused" if fused else "k-split"
    out["route"]["tensor_peak"] = f"bf16 burst {bf16} TFLOP/s (measured)"
    out["note"] = ("device time per call from CUDA events inside the timed step; hbm_frac of the measured "
                   f"copy bandwidth {hbm} GB/s, tensor_frac of the measured bf16 burst (route) or 2x it (FP8 GEMMs)")
    return out


TRAIN_METRIC = "MoE layer forward+backward tokens/s; FP8 weight-gradient GEMM TFLOP/s & % of roofline (1 B300)"


def run_train(args):
    """--backward: a training step of the layer (forward, bias update, backward) on one GPU."""
    import torch

    import __graft_entry__
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.configs import CONFIGS, PROFILE_CONFIGS
    from sparse_moe_layer_13_b300.layer import MoELayer

    torch.cuda.set_device(0)
    __graft_entry__.build()
    cfg = {**CONFIGS, **PROFILE_CONFIGS}[args.config]
    layer = MoELayer(cfg, "cuda", scale_rule=args.scales, backward=True)
    x = inputs.gen_x(cfg, "cuda")
    dy = inputs.gen_dy(cfg, "cuda")
    names = ("gemm1", "gemm2")
    bnames = ("dgrad2", "recompute", "dgrad1", "wgrad2", "wgrad1")
    K = args.steps

    def _step(i=None, ev=None):
        layer.forward(x, update_bias=False, events=None if ev is None else {n: ev[n][i] for n in names})
        binding.bias_update(cfg.E, cfg.T, cfg.K, layer.counts, cfg.gamma, layer.bias)
        return layer.backward(x, dy, events=None if ev is None else {n: ev[n][i] for n in bnames})

    for _ in range(args.warmup):
        _step()
    torch.cuda.synchronize()
    binding.check_device_status()
    ev = {n: [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
              for _ in range(K)] for n in names + bnames}
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(K):
                _step(i, ev)
        graph.replay()
        torch.cuda.synchronize()
        binding.check_device_status()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        torch.cuda.synchronize()
        t0.record()
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                _step(i, ev)
        t1.record()
        torch.cuda.synchronize()
    binding.check_device_status()
    ms = t0.elapsed_time(t1) / K
    kt = {n: statistics.mean(a.elapsed_time(b) for a, b in ev[n]) for n in names + bnames}

    # end to end: x and dy from pinned host memory, dx back, every step (serial copies)
    xh, dyh = x.cpu().pin_memory(), dy.cpu().pin_memory()
    dxh = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    xd, dyd = torch.empty_like(x), torch.empty_like(dy)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K):
        xd.copy_(xh, non_blocking=True)
        dyd.copy_(dyh, non_blocking=True)
        layer.forward(xd, update_bias=False)
        binding.bias_update(cfg.E, cfg.T, cfg.K, layer.counts, cfg.gamma, layer.bias)
        dxh.copy_(layer.backward(xd, dyd)["dx"], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K

    hbm, bf16, bf16_s, src = _peaks()
    fp8_peak = 2.0 * bf16
    clock_summary = clocks.summary()
    roof_peak, roof_src = _fp8_peak(bf16, bf16_s, src, clock_summary)
    R, d, I, E1 = cfg.rows, cfg.d, cfg.I, cfg.E + 1
    # weight gradient of W1|W3: 2 * rows * 2I * d FLOPs; its bytes: the FP32 gradient written
    # (E+1) * 2I * d * 4, plus both transposed E4M3 operands and their 128x1 scales read once
    width = binding.q1_width(E1, R)
    w1_flops = 2.0 * R * 2 * I * d
    w1_bytes = E1 * 2 * I * d * 4 + (2 * I + d) * width * (1 + 4 / 128)
    w1_ms = kt["wgrad1"]
    t_tensor, t_hbm = w1_flops / (roof_peak * 1e12), w1_bytes / (hbm * 1e9)
    if t_hbm > t_tensor:
        roof = {"kernel": "grouped_wgrad_fp8 (dW1|dW3)", "bound": "hbm",
                "achieved": round(w1_bytes / (w1_ms * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(w1_bytes / (w1_ms * 1e-3) / 1e9 / hbm, 4), "traffic": None,
                "algorithmic_bytes": round(w1_bytes), "peak_source": f"{src}: HBM copy bandwidth"}
    else:
        roof = {"kernel": "grouped_wgrad_fp8 (dW1|dW3)", "bound": "tensor",
                "achieved": round(w1_flops / (w1_ms * 1e-3) / 1e12, 1), "peak": round(roof_peak, 1),
                "unit": "TFLOP/s", "frac": round(w1_flops / (w1_ms * 1e-3) / 1e12 / roof_peak, 4), "traffic": None,
                "peak_source": roof_src}
    roof["tensor_frac"] = round(w1_flops / (w1_ms * 1e-3) / 1e12 / fp8_peak, 4)
    roof["hbm_frac"] = round(w1_bytes / (w1_ms * 1e-3) / 1e9 / hbm, 4)
    f1, f2 = cfg.gemm_flops()
    # algorithmic backward FLOPs: data and weight gradients of both GEMMs (the recomputation of
    # the gate/up pre-activations, another f1, is work done but not counted)
    bwd_flops = 2 * f1 + 2 * f2
    out = {
        "metric": TRAIN_METRIC, "value": round(cfg.T / (ms * 1e-3), 1), "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) x and dy, N(0,1/d) weights, random init)",
        "config": {"workload": f"{cfg.name} training step: T={cfg.T} d={cfg.d} E={cfg.E}+1 I={cfg.I} K={cfg.K} "
                               f"G={cfg.G} M={cfg.M}", "scale_rule": args.scales, "parallelism": "dp1",
                   "launch": "one CUDA graph of the K steps" if graph is not None else "eager launches",
                   "l2": "inputs exceed L2 (x, dy, weights and gradients read or written every step), no flush"},
        "layer_tflops": round((cfg.flops() + bwd_flops) / (ms * 1e-3) / 1e12, 1),
        "kernels_ms": {n: round(v, 4) for n, v in kt.items()},
        "roofline": roof,
        "e2e": {"value": round(cfg.T / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": 2 * cfg.T * d * 2,
                "d2h_bytes_per_step": cfg.T * d * 2},
        "gpu_launches": K * (layer.launches_per_forward + layer.launches_per_backward),
        "clocks": clock_summary,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_train(cfg, n_tokens=args.cpu_tokens)
    print(json.dumps(out), flush=True)


def cpu_baseline_train(cfg, n_tokens: int):
    """The FP64 oracle's training step as it stands, on a sample of n_tokens tokens: the
    layer forward of the sample and its backward down to the input gradient (the expert
    rows of the sampled tokens, router gradient included; weight gradients, which sum
    over every row of an expert, are not in the sample). Weight quantisation untimed."""
    import numpy as np
    import torch

    from oracle.backward import dequant_expert, layer_backward
    from oracle.layer import Layer
    from oracle.parallel import quantize_experts
    from oracle.route import affinity, route as oracle_route
    from sparse_moe_layer_13_b300 import inputs

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = inputs.gen_x(cfg, dev).float().cpu().numpy()
    dy = inputs.gen_dy(cfg, dev).float().cpu().numpy()
    Wr = inputs.gen_router(cfg, dev).cpu().numpy()
    b = inputs.gen_bias(cfg, dev).cpu().numpy()
    rng = np.random.default_rng(4321)
    tok = np.sort(rng.choice(cfg.T, n_tokens, replace=False))
    idx, _, _ = oracle_route(x[tok], Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)
    need = sorted(set(idx.ravel().tolist()) | {cfg.E})
    ex = quantize_experts((e, *(w.cpu().numpy() for w in inputs.gen_expert(cfg, e, dev))) for e in need)
    deq = {e: dequant_expert(w) for e, w in ex.items()}
    layer = Layer(cfg, Wr, b, None, experts=ex)
    sub = type("Sample", (), {"T": n_tokens, "d": cfg.d, "E": cfg.E, "I": cfg.I, "K": cfg.K})()
    t = time.perf_counter()
    fwd = layer.forward(x[tok])
    s_sel = np.take_along_axis(affinity(x[tok], Wr), fwd["idx"], axis=1)
    layer_backward(sub, x[tok], dy[tok], Wr, fwd["idx"], s_sel, lambda e: deq[e], tokens=range(n_tokens))
    dt = time.perf_counter() - t
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except ImportError:
        blas = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or os.cpu_count())
    return {"value": round(n_tokens / dt, 4), "unit": UNIT, "cores": blas, "kind": "oracle",
            "sample": f"{n_tokens} tokens of the {cfg.name} batch: layer forward and backward to the input "
                      f"gradient (router gradient included, weight gradients not) in FP64; weight "
                      f"quantisation untimed",
            "host_cpus": os.cpu_count()}


def e2e_pipelined(cfg, layer, x, K, hook, binding, T_all):
    """Milliseconds per step of K forwards fed from and drained to pinned host memory."""
    import torch
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    xh = [x.cpu().pin_memory() for _ in range(2)]
    yh = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(x) for _ in range(2)]
    x_ready = [torch.cuda.Event() for _ in range(2)]
    x_free = [torch.cuda.Event() for _ in range(2)]
    y_ready = [torch.cuda.Event() for _ in range(2)]
    y_free = [torch.cuda.Event() for _ in range(2)]
    for i in range(2):
        x_free[i].record(comp)
        y_free[i].record(comp)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(x_free[b])
            xd[b].copy_(xh[b], non_blocking=True)
            x_ready[b].record(h2d)

    e0.record(comp)
    upload(0)
    for i in range(K):
        b = i % 2
        if i + 1 < K:
            upload(i + 1)                      # overlaps this step's compute
        comp.wait_event(x_ready[b])
        comp.wait_event(y_free[b])
        layer.forward(xd[b], update_bias=False, out=yd[b])
        x_free[b].record(comp)
        if hook is not None:
            hook(layer.counts)
        binding.bias_update(cfg.E, T_all, cfg.K, layer.counts, cfg.gamma, layer.bias)
        y_ready[b].record(comp)
        with torch.cuda.stream(d2h):           # overlaps the next step's compute
            d2h.wait_event(y_ready[b])
            yh[b].copy_(yd[b], non_blocking=True)
            y_free[b].record(d2h)
    comp.wait_stream(d2h)
    e1.record(comp)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def balancing_loop(cfg, layer, dev, binding, inputs, dp):
    """cfg.skew_steps steps of (route with loads -> end-of-step bias update) on fresh
    batches; returns the max/mean and min/mean expert load seen at each step."""
    import torch
    mx, mn = [], []
    T_all = dp.global_tokens(cfg.T)
    for step in range(cfg.skew_steps):
        x = inputs.gen_x(cfg, dev, step=1000 + step)
        binding.route_planes(cfg, x, layer.planes, layer.bias, layer.logit_offset, layer.ws, layer.idx, layer.gate,
                             layer.counts)
        dp.allreduce_load(layer.counts)
        binding.bias_update(cfg.E, T_all, cfg.K, layer.counts, cfg.gamma, layer.bias)
        c = layer.counts.cpu().numpy().astype("float64")
        mean = T_all * cfg.K / cfg.E
        mx.append(round(float(c.max() / mean), 3))
        mn.append(round(float(c.min() / mean), 3))
    torch.cuda.synchronize()
    return {"steps": cfg.skew_steps, "gamma": cfg.gamma, "zipf_s": cfg.zipf_s, "zipf_c": cfg.zipf_c,
            "max_over_mean": mx, "min_over_mean": mn}


def cpu_baseline(cfg, n_tokens: int, steps: int):
    """The FP64 oracle as it stands, on a sample of n_tokens tokens of the workload.

    Weight quantisation is set-up on both sides and is not timed (here it
    runs in parallel worker processes); each step times Layer.forward on a
    fresh sample of tokens drawn from the same seeded batch.
    """
    import numpy as np
    import torch

    from oracle.layer import Layer
    from oracle.parallel import quantize_experts
    from oracle.route import route as oracle_route
    from sparse_moe_layer_13_b300 import inputs

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = inputs.gen_x(cfg, dev).float().cpu().numpy()
    Wr = inputs.gen_router(cfg, dev).cpu().numpy()
    b = inputs.gen_bias(cfg, dev).cpu().numpy()
    rng = np.random.default_rng(1234)
    samples = [np.sort(rng.choice(cfg.T, n_tokens, replace=False)) for _ in range(steps)]
    idx, _, _ = oracle_route(x[np.concatenate(samples)], Wr, b, cfg.G, cfg.M, cfg.K, cfg.gk)
    need = sorted(set(idx.ravel().tolist()) | {cfg.E})
    ex = quantize_experts((e, *(w.cpu().numpy() for w in inputs.gen_expert(cfg, e, dev))) for e in need)
    layer = Layer(cfg, Wr, b, None, experts=ex)
    threads = torch.get_num_threads()
    t = time.perf_counter()
    for s in samples:
        layer.forward(x[s])
    dt = time.perf_counter() - t
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except ImportError:      # OpenBLAS uses every host core unless told otherwise
        blas = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or os.cpu_count())
    return {"value": round(n_tokens * steps / dt, 4), "unit": UNIT, "cores": blas, "kind": "oracle",
            "sample": f"{n_tokens * steps} tokens of the {cfg.name} batch (whole layer per token: route, "
                      f"quantise, {cfg.K}+1 expert FFNs in FP64, combine); weight quantisation untimed",
            "host_cpus": os.cpu_count(), "torch_threads": threads}


def run_reference(args):
    """--impl reference: the oracle itself, timed on the host cores, same metric and config."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from sparse_moe_layer_13_b300.configs import CONFIGS
    cfg = CONFIGS[args.config]
    n = max(1, args.ref_tokens)
    # warm-up steps run the same sampled forward untimed inside cpu_baseline's single pass
    cb = cpu_baseline(cfg, n_tokens=n, steps=max(1, args.steps))
    ms = 1e3 * n / cb["value"]
    out = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 0,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E}+1 I={cfg.I} K={cfg.K} G={cfg.G} M={cfg.M}"},
           "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
           "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_fp8_peak(args):
    """--fp8-peak: dense E4M3 GEMM throughput of the vendor library on this GPU (torch._scaled_mm,
    8192^3, per-tensor unit scales, bf16 output), best of 10 timed with CUDA events after 3
    warm-ups, with the SM clock sampled meanwhile. A measured context figure for the FP8
    roofline denominators; the reported fractions keep the bf16 figure of MEASURED_PEAKS.json."""
    import torch
    torch.cuda.set_device(0)
    n = 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    a = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn).t()   # column-major operand
    one = torch.ones((), device="cuda")
    for _ in range(3):
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    best = float("inf")
    with ClockSampler(0) as clocks:
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
    tf = 2.0 * n ** 3 / (best * 1e-3) / 1e12
    _, bf16, _, src = _peaks()
    print(json.dumps({"measurement": "fp8 e4m3 dense GEMM peak (torch._scaled_mm 8192^3, best of 10)",
                      "tflops": round(tf, 1), "ms": round(best, 4), "bf16_burst_tflops": bf16,
                      "ratio_to_bf16": round(tf / bf16, 3), "clocks": clocks.summary()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="full")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=4)
    ap.add_argument("--ref-tokens", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph of the K steps")
    ap.add_argument("--scales", default="fp32", choices=["fp32", "pow2"],
                    help="pow2: power-of-two 1x128 / 128x128 scales and the block-scaled GEMMs")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step (forward, bias update, backward) instead of the forward")
    ap.add_argument("--fp8-peak", action="store_true",
                    help="measure the vendor library's dense E4M3 GEMM rate (8192^3) and exit")
    args = ap.parse_args()
    if args.fp8_peak:
        run_fp8_peak(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.backward:
        run_train(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
