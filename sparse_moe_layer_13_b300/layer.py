"""DeepSeekMoE layer forward on one B300, chaining the C-ABI calls.

《DeepSeek-V3 Technical Report》深度解读报告 §2.2-§2.4 and "DeepSeek-V3的MoE架构
设计革新" §2 describe the layer; this module only owns device buffers and
calls, in order: moe_route_planes -> moe_permute (row order only) ->
moe_quant_fp8_1x128_scatter (tokens quantised straight into grouped rows) ->
moe_grouped_gemm_fp8 (gate/up + SwiGLU + requantisation) ->
moe_grouped_gemm_fp8 (down) -> moe_combine -> moe_bias_update. Expert E (the
last group) is the shared expert.

token_rows picks how the gate/up GEMM gets its grouped token rows:
  "scatter"  the quantiser writes them (default, least traffic);
  "copy"     quantise in token order, then moe_permute gathers a copy;
  "gather"   quantise in token order and let the GEMM fetch rows by index
             (moe_grouped_gemm_fp8_gather: no grouped copy, (K+1)*T*d fewer
             bytes of device memory, slower GEMM).
All three give bit-identical results.

scale_rule "pow2" quantises x, the weights and h with power-of-two scales and
runs both grouped GEMMs on the block-scaled MMA (moe_grouped_gemm_fp8_mx).
"""
from __future__ import annotations

import torch

from . import binding as B
from . import dp, inputs
from .configs import MoEConfig


class ExpertWeights:
    """FP8 expert weights on the device, built from the seeded generator, with
    128x128 scales under `scale_rule` ("fp32" or "pow2").

    q13 u8 [E+1][2I][d] (SwiGLU layout), s13 f32 [E+1][2I/128][d/128],
    q2  u8 [E+1][d][I],                  s2  f32 [E+1][d/128][I/128].
    With backward=True also the transposed blocks the data gradients use:
    q13T u8 [E+1][d][2I] (K order [W1 | W3]), s13T f32 [E+1][d/128][2I/128],
    q2T  u8 [E+1][Ip][d] (rows I..Ip-1 zero, Ip = I rounded up to 256),
                         s2T f32 [E+1][Ip/128][d/128].
    """

    def __init__(self, cfg: MoEConfig, device="cuda", chunk: int = 16, scale_rule: str = "fp32",
                 backward: bool = False):
        E1, I, d = cfg.E + 1, cfg.I, cfg.d
        self.scale_rule = scale_rule
        self.backward = backward
        self.q13 = torch.empty(E1, 2 * I, d, dtype=torch.uint8, device=device)
        self.s13 = torch.empty(E1, 2 * I // 128, d // 128, dtype=torch.float32, device=device)
        self.q2 = torch.empty(E1, d, I, dtype=torch.uint8, device=device)
        self.s2 = torch.empty(E1, d // 128, I // 128, dtype=torch.float32, device=device)
        if backward:
            Ip = (I + 255) // 256 * 256
            self.q13T = torch.empty(E1, d, 2 * I, dtype=torch.uint8, device=device)
            self.s13T = torch.empty(E1, d // 128, 2 * I // 128, dtype=torch.float32, device=device)
            self.q2T = torch.zeros(E1, Ip, d, dtype=torch.uint8, device=device)
            self.s2T = torch.zeros(E1, Ip // 128, d // 128, dtype=torch.float32, device=device)
        for e0 in range(0, E1, chunk):
            e1 = min(E1, e0 + chunk)
            ws = [inputs.gen_expert(cfg, e, device) for e in range(e0, e1)]
            w1 = torch.stack([w[0] for w in ws])
            w3 = torch.stack([w[1] for w in ws])
            w2 = torch.stack([w[2] for w in ws])
            del ws
            q1, s1 = B.quant_128x128(w1, rule=scale_rule)
            q3, s3 = B.quant_128x128(w3, rule=scale_rule)
            B.pack_w13(q1, s1, q3, s3, self.q13[e0:e1], self.s13[e0:e1])
            B.quant_128x128(w2, self.q2[e0:e1], self.s2[e0:e1], rule=scale_rule)
            if backward:
                B.transpose_fp8_blocks(q1, s1, self.q13T[e0:e1], self.s13T[e0:e1], offset=0)
                B.transpose_fp8_blocks(q3, s3, self.q13T[e0:e1], self.s13T[e0:e1], offset=I)
                B.transpose_fp8_blocks(self.q2[e0:e1], self.s2[e0:e1], self.q2T[e0:e1], self.s2T[e0:e1])
            del w1, w3, w2, q1, q3


class MoELayer:
    """One layer instance: router weight, selection bias, expert weights, buffers."""

    def __init__(self, cfg: MoEConfig, device="cuda", weights: ExpertWeights | None = None,
                 logit_offset: torch.Tensor | None = None, token_rows: str = "scatter", scale_rule: str = "fp32",
                 backward: bool = False):
        if token_rows not in ("scatter", "copy", "gather"):
            raise ValueError(f"token_rows: {token_rows!r}")
        if scale_rule not in ("fp32", "pow2"):
            raise ValueError(f"scale_rule: {scale_rule!r}")
        if scale_rule == "pow2" and token_rows == "gather":
            raise ValueError("the block-scaled GEMM reads grouped rows; use token_rows 'scatter' or 'copy'")
        self.cfg = cfg
        self.token_rows = token_rows
        self.scale_rule = scale_rule
        self.block_scaled = scale_rule == "pow2"
        self.device = device
        self.Wr = inputs.gen_router(cfg, device)
        self.planes = B.router_planes(self.Wr)        # redo with refresh_router() when Wr changes
        self.bias = inputs.gen_bias(cfg, device)
        self.logit_offset = logit_offset
        self.w = ExpertWeights(cfg, device, scale_rule=scale_rule, backward=backward) if weights is None else weights
        self._bwd = None
        if self.w.scale_rule != scale_rule:
            raise ValueError("the expert weights were quantised with another scale rule")
        T, K, E, d, I = cfg.T, cfg.K, cfg.E, cfg.d, cfg.I
        R = cfg.rows
        z = lambda *s, dt: torch.empty(*s, dtype=dt, device=device)  # noqa: E731
        self.ws = z(B.workspace_size(cfg), dt=torch.uint8)
        self.idx = z(T, K, dt=torch.int32)
        self.gate = z(T, K, dt=torch.float32)
        self.counts = z(E, dt=torch.int32)
        grouped = token_rows != "gather"
        self.xq = z(T, d, dt=torch.uint8) if token_rows != "scatter" else None
        self.xs = z(T, d // 128, dt=torch.float32) if token_rows != "scatter" else None
        self.xq_perm = z(R, d, dt=torch.uint8) if grouped else None
        self.xs_perm = z(R, d // 128, dt=torch.float32) if grouped else None
        self.perm = {
            "offsets": z(E + 2, dt=torch.int32), "counts": None,
            "sorted_token": z(R, dt=torch.int32), "row_of": z(T, K, dt=torch.int32),
            "xq_perm": self.xq_perm if token_rows == "copy" else None,
            "xs_perm": self.xs_perm if token_rows == "copy" else None,
        }
        self.hq = z(R, I, dt=torch.uint8)
        self.hs = z(R, I // 128, dt=torch.float32)
        self.out = z(R, d, dt=torch.bfloat16)          # routed rows (the shared rows stay unused)
        self.out_shared = z(T, d, dt=torch.float32)
        self.y = z(T, d, dt=torch.bfloat16)

    def forward(self, x: torch.Tensor, residual: bool = False, update_bias: bool = True,
                gamma: float | None = None, counts_hook=None, load_tokens: int | None = None, events=None,
                out: torch.Tensor | None = None) -> torch.Tensor:
        """One layer forward on the current stream.

        counts_hook(counts) runs before the bias update (e.g. dp.allreduce_load,
        which sums the expert load over data-parallel ranks); load_tokens is
        the number of tokens those counts then cover, against whose mean load
        T*K/E the update judges each expert. It defaults to this layer's T
        without a hook and to dp.global_tokens(T) with one (every rank of the
        default group holding T tokens). events, if given, is a dict of
        name -> (start, end) torch.cuda.Event pairs recorded around the calls
        "route" (router with loads), "permute" (row order), "quant" (quantise
        into grouped rows, token_rows "scatter"), "gemm1" (gate/up + SwiGLU),
        "gemm2" (down) and "combine"; out, if given, receives y (bf16 [T][d])
        instead of the layer's own buffer.
        """
        c = self.cfg
        ev = events or {}

        def mark(name, i):
            if name in ev:
                ev[name][i].record()

        mark("route", 0)
        B.route_planes(c, x, self.planes, self.bias, self.logit_offset, self.ws, self.idx, self.gate, self.counts)
        mark("route", 1)
        mode = self.token_rows
        rule = self.scale_rule
        if mode != "scatter":
            B.quant_1x128(x, self.xq, self.xs, rule=rule)
        mark("permute", 0)
        B.permute(c, self.idx, self.xq, self.xs, self.ws, self.perm, gather_rows=mode == "copy")
        mark("permute", 1)
        if mode == "scatter":
            mark("quant", 0)
            B.quant_1x128_scatter(c, x, self.perm["row_of"], self.xq_perm, self.xs_perm, rule=rule)
            mark("quant", 1)
        if "gemm1" in ev:
            ev["gemm1"][0].record()
        if mode == "gather":
            B.grouped_gemm_fp8(self.perm["offsets"], self.xq, self.xs, self.w.q13, self.w.s13, B.MOE_EPI_SWIGLU_FP8,
                               self.hq, self.hs, row_index=self.perm["sorted_token"])
        else:
            B.grouped_gemm_fp8(self.perm["offsets"], self.xq_perm, self.xs_perm, self.w.q13, self.w.s13,
                               B.MOE_EPI_SWIGLU_FP8, self.hq, self.hs, block_scaled=self.block_scaled)
        if "gemm1" in ev:
            ev["gemm1"][1].record()
        if "gemm2" in ev:
            ev["gemm2"][0].record()
        B.grouped_gemm_fp8(self.perm["offsets"], self.hq, self.hs, self.w.q2, self.w.s2, B.MOE_EPI_BF16_F32_LAST,
                           self.out, self.out_shared, block_scaled=self.block_scaled)
        if "gemm2" in ev:
            ev["gemm2"][1].record()
        TK = c.T * c.K
        y = self.y if out is None else out
        mark("combine", 0)
        B.combine(c, self.out[:TK], self.out_shared, self.perm["row_of"], self.gate, x if residual else None, y)
        mark("combine", 1)
        if update_bias:
            self.end_of_step(gamma, counts_hook, load_tokens)
        return y

    def refresh_router(self):
        """Re-splits the router weight into the bf16 planes the router reads (after Wr changed)."""
        B.router_planes(self.Wr, self.planes)

    def end_of_step(self, gamma: float | None = None, counts_hook=None, load_tokens: int | None = None):
        """The end-of-step bias update on the last routing's expert load
        (《DeepSeek-V3 Technical Report》深度解读报告 §2.3): counts_hook(counts)
        first (e.g. the data-parallel all-reduce), then every bias moves by
        gamma towards the mean load of the tokens the counts cover."""
        c = self.cfg
        if counts_hook is not None:
            counts_hook(self.counts)
            T = dp.global_tokens(c.T) if load_tokens is None else load_tokens
        else:
            T = c.T if load_tokens is None else load_tokens
        B.bias_update(c.E, T, c.K, self.counts, c.gamma if gamma is None else gamma, self.bias)

    def backward(self, x: torch.Tensor, dy: torch.Tensor, events=None) -> dict:
        """Gradients of the last forward (on x) for upstream gradient dy (bf16 [T][d]),
        with the chosen experts held fixed, on the current stream.

        Reads what the forward left: routing, grouped rows, the quantised x and
        h, the routed outputs and the router logits in the workspace; call it
        before the next forward. Needs weights built with backward=True and
        token_rows "scatter" or "copy". Returns device tensors (reused by the
        next call):
          dx   bf16 [T][d]
          dWr  f32  [E][d]
          dW13 f32  [E+1][2I][d]  in the q13 (SwiGLU tile) row layout
          dW2T f32  [E+1][I][d]   the down projection's gradient, transposed
          dgate, dz f32 [T][K]    gate and router-logit gradients
        Every FP8 GEMM runs on the FP32-scale tensor-core kernels under the
        layer's scale rule. events, if given, maps "dgrad2", "recompute",
        "dgrad1", "wgrad2", "wgrad1" to (start, end) event pairs recorded
        around those GEMMs.
        """
        c = self.cfg
        if not getattr(self.w, "backward", False):
            raise ValueError("expert weights were built without backward=True")
        if self.token_rows == "gather":
            raise ValueError("the backward pass reads the grouped token rows; use token_rows 'scatter' or 'copy'")
        B._need(dy, torch.bfloat16, "dy", (c.T, c.d))
        bw = self._bwd_buffers()
        rule = self.scale_rule
        T, K, E, d, I = c.T, c.K, c.E, c.d, c.I
        R = c.rows
        offs, st, ro = self.perm["offsets"], self.perm["sorted_token"], self.perm["row_of"]
        B.combine_backward(c, dy, self.out, ro, self.gate, bw["dOq"], bw["dOs"], bw["row_gate"], bw["dgate"], rule)
        B.route_backward(c, self.idx, bw["dgate"], self.ws, bw["dz"], self.logit_offset)
        B.router_wgrad(c, x, offs[:E + 1], st, ro, bw["dz"], bw["dWr"])
        ev = events or {}

        def mark(name, i):
            if name in ev:
                ev[name][i].record()

        mark("dgrad2", 0)
        B.grouped_gemm_fp8(offs, bw["dOq"], bw["dOs"], self.w.q2T, self.w.s2T, B.MOE_EPI_F32, bw["dh"])
        mark("dgrad2", 1)
        mark("recompute", 0)
        B.grouped_gemm_fp8(offs, self.xq_perm, self.xs_perm, self.w.q13, self.w.s13, B.MOE_EPI_GATEUP_F32, bw["ab"])
        mark("recompute", 1)
        B.swiglu_backward(bw["ab"], bw["dh"], bw["dabq"], bw["dabs"], rule)
        mark("dgrad1", 0)
        B.grouped_gemm_fp8(offs, bw["dabq"], bw["dabs"], self.w.q13T, self.w.s13T, B.MOE_EPI_BF16_F32_LAST,
                           bw["dxr"], bw["dxs"])
        mark("dgrad1", 1)
        B.dx_combine(c, bw["dxr"], bw["dxs"], ro, self.idx, bw["dz"], self.Wr, bw["dx"])
        B.quant_128x1(offs, R, d, rule, bw["oT"], bw["oS"], bf16_rows=(dy, st, bw["row_gate"]))
        B.quant_128x1(offs, R, I, rule, bw["hT"], bw["hS"], fp8=(self.hq, self.hs))
        B.quant_128x1(offs, R, 2 * I, rule, bw["gT"], bw["gS"], f32=bw["ab"])
        B.quant_128x1(offs, R, d, rule, bw["xT"], bw["xS"], fp8=(self.xq_perm, self.xs_perm))
        mark("wgrad2", 0)
        B.grouped_wgrad_fp8(offs, R, bw["hT"], bw["hS"], bw["oT"], bw["oS"], bw["dW2T"])
        mark("wgrad2", 1)
        mark("wgrad1", 0)
        B.grouped_wgrad_fp8(offs, R, bw["gT"], bw["gS"], bw["xT"], bw["xS"], bw["dW13"])
        mark("wgrad1", 1)
        return {k: bw[k] for k in ("dx", "dWr", "dW13", "dW2T", "dgate", "dz")}

    # library kernel launches per backward: combine 1, route 1, router weight 1, GEMMs 5,
    # SwiGLU 1, input gradient 1, 128x1 quantisers 4
    launches_per_backward = 14

    def _bwd_buffers(self) -> dict:
        if getattr(self, "_bwd", None) is None:
            c = self.cfg
            T, K, E, d, I = c.T, c.K, c.E, c.d, c.I
            R = c.rows
            Ip = self.w.q2T.shape[1]
            W = B.q1_width(E + 1, R)
            z = lambda *s, dt: torch.empty(*s, dtype=dt, device=self.device)  # noqa: E731
            f32, u8 = torch.float32, torch.uint8
            self._bwd = {
                "dOq": z(R, d, dt=u8), "dOs": z(R, d // 128, dt=f32), "row_gate": z(R, dt=f32),
                "dgate": z(T, K, dt=f32), "dz": z(T, K, dt=f32), "dWr": z(E, d, dt=f32),
                "dh": z(R, Ip, dt=f32), "ab": z(R, 2 * I, dt=f32),
                "dabq": z(R, 2 * I, dt=u8), "dabs": z(R, 2 * I // 128, dt=f32),
                "dxr": z(R, d, dt=torch.bfloat16), "dxs": z(T, d, dt=f32), "dx": z(T, d, dt=torch.bfloat16),
                "oT": z(d, W, dt=u8), "oS": z(W // 128, d, dt=f32),
                "hT": z(I, W, dt=u8), "hS": z(W // 128, I, dt=f32),
                "gT": z(2 * I, W, dt=u8), "gS": z(W // 128, 2 * I, dt=f32),
                "xT": z(d, W, dt=u8), "xS": z(W // 128, d, dt=f32),
                "dW2T": z(E + 1, I, d, dt=f32), "dW13": z(E + 1, 2 * I, d, dt=f32),
            }
        return self._bwd

    def balance_loss(self, seq_len: int, alpha: float, stats: bool = False):
        """Sequence-wise balance loss of the last forward's routing (loss per sequence of
        seq_len tokens, and f, P [sequences][E] if stats); reads the router logits that the
        forward left in the workspace, so call it before the next forward."""
        return B.balance_loss(self.cfg, self.idx, self.ws, seq_len, alpha, self.logit_offset, stats)

    def capture(self, x: torch.Tensor, steps: int = 1, events=None, **forward_kw) -> torch.cuda.CUDAGraph:
        """Records `steps` forwards of x into a CUDA graph; graph.replay() reruns them on
        whatever x (a fixed device buffer) holds then, without per-launch host work.

        forward_kw go to forward() (residual, update_bias, gamma, out); events, if given, is a
        list of per-step event dicts as forward() takes, recorded inside the graph (create them
        with torch.cuda.Event(enable_timing=True, external=True) to time replays). Every
        library kernel must have run once before (one plain forward): a first launch sets
        kernel attributes, which a capture does not record.
        """
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(steps):
                self.forward(x, events=None if events is None else events[i], **forward_kw)
        return graph

    # library kernel launches per forward: route 3 (fused router, histogram, scan) or 4 on the
    # K-split path (logits, selection, histogram, scan), quantise 1, permute 3 (+1 row gather
    # for "copy"), grouped GEMMs 2, combine 1, bias update 1
    @property
    def route_fused(self) -> bool:
        """Whether moe_route_planes' automatic choice takes the fused router for this layer."""
        c = self.cfg
        sms = torch.cuda.get_device_properties(torch.device(self.device)).multi_processor_count
        return c.E <= 256 and 2 * ((c.T + 127) // 128) >= sms

    @property
    def launches_per_forward(self) -> int:
        return (3 if self.route_fused else 4) + 8 + int(self.token_rows == "copy")
