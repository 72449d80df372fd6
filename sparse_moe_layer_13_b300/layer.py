"""DeepSeekMoE layer forward on one B300, chaining the C-ABI calls.

《DeepSeek-V3 Technical Report》深度解读报告 §2.2-§2.4 and "DeepSeek-V3的MoE架构
设计革新" §2 describe the layer; this module only owns device buffers and
calls, in order: moe_route -> moe_permute (row order only) ->
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
from . import inputs
from .configs import MoEConfig


class ExpertWeights:
    """FP8 expert weights on the device, built from the seeded generator, with
    128x128 scales under `scale_rule` ("fp32" or "pow2").

    q13 u8 [E+1][2I][d] (SwiGLU layout), s13 f32 [E+1][2I/128][d/128],
    q2  u8 [E+1][d][I],                  s2  f32 [E+1][d/128][I/128].
    """

    def __init__(self, cfg: MoEConfig, device="cuda", chunk: int = 16, scale_rule: str = "fp32"):
        E1, I, d = cfg.E + 1, cfg.I, cfg.d
        self.scale_rule = scale_rule
        self.q13 = torch.empty(E1, 2 * I, d, dtype=torch.uint8, device=device)
        self.s13 = torch.empty(E1, 2 * I // 128, d // 128, dtype=torch.float32, device=device)
        self.q2 = torch.empty(E1, d, I, dtype=torch.uint8, device=device)
        self.s2 = torch.empty(E1, d // 128, I // 128, dtype=torch.float32, device=device)
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
            del w1, w3, w2, q1, q3


class MoELayer:
    """One layer instance: router weight, selection bias, expert weights, buffers."""

    def __init__(self, cfg: MoEConfig, device="cuda", weights: ExpertWeights | None = None,
                 logit_offset: torch.Tensor | None = None, token_rows: str = "scatter", scale_rule: str = "fp32"):
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
        self.bias = inputs.gen_bias(cfg, device)
        self.logit_offset = logit_offset
        self.w = ExpertWeights(cfg, device, scale_rule=scale_rule) if weights is None else weights
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
                gamma: float | None = None, counts_hook=None, events=None, out: torch.Tensor | None = None) -> torch.Tensor:
        """One layer forward on the current stream.

        counts_hook(counts) runs before the bias update (e.g. an all-reduce of
        the expert load across data-parallel ranks); events, if given, is a
        dict of name -> (start, end) torch.cuda.Event pairs recorded around
        the two grouped GEMMs ("gemm1", "gemm2"); out, if given, receives y
        (bf16 [T][d]) instead of the layer's own buffer.
        """
        c = self.cfg
        ev = events or {}
        B.route(c, x, self.Wr, self.bias, self.logit_offset, self.ws, self.idx, self.gate, self.counts)
        mode = self.token_rows
        rule = self.scale_rule
        if mode != "scatter":
            B.quant_1x128(x, self.xq, self.xs, rule=rule)
        B.permute(c, self.idx, self.xq, self.xs, self.ws, self.perm, gather_rows=mode == "copy")
        if mode == "scatter":
            B.quant_1x128_scatter(c, x, self.perm["row_of"], self.xq_perm, self.xs_perm, rule=rule)
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
        B.combine(c, self.out[:TK], self.out_shared, self.perm["row_of"], self.gate, x if residual else None, y)
        if update_bias:
            if counts_hook is not None:
                counts_hook(self.counts)
            B.bias_update(c.E, c.T, c.K, self.counts, c.gamma if gamma is None else gamma, self.bias)
        return y

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

    # library kernel launches per forward: route 5 (weight split, logits, selection, histogram,
    # scan), quantise 1, permute 3 (+1 row gather for "copy"), grouped GEMMs 2, combine 1,
    # bias update 1
    @property
    def launches_per_forward(self) -> int:
        return 13 + int(self.token_rows == "copy")
