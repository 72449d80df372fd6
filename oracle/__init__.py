"""FP64 CPU oracle for the DeepSeekMoE layer (forward and backward).

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously correct
restatement of what the layer computes, used to check the CUDA library.
Only the test suite, the package smoke check and the benchmark's CPU
baseline leg may import it; the CUDA path never does, and it shares no
code with the CUDA path (only the seeded input generator feeds both).

Passages followed (page title, section):

* 《DeepSeek-V3 Technical Report》深度解读报告 §2.2 DeepSeekMoE: the layer
  output is the input plus the shared expert FFN plus the gate-weighted
  routed expert FFNs; gates are sigmoid affinities renormalised over the
  chosen experts.
* same page §2.3 Auxiliary-Loss-Free Load Balancing: a per-expert bias is
  added to the affinity for top-K choice only; gates come from the raw
  affinity; at each step's end overloaded experts' bias drops by gamma and
  underloaded experts' bias rises by gamma, judged on the whole batch.
* same page §2.4 Node-Limited Routing: a token reaches at most M nodes,
  chosen by the sum of the highest affinities of the experts on each node;
  no token is dropped.
* "DeepSeek-V3的MoE架构设计革新" (devpress blog) §2 FP8 training, items 1-2:
  weights quantised per 128x128 block, activations per 1x128 tile, FP32
  accumulation every 128 elements of the contraction.
* "DeepSeek-V3技术解析：MoE、FP8与MLA如何突破大模型推理瓶颈" §3.1 and §6.2:
  FP8 values use E4M3, whose largest finite value is 448.

Modules: e4m3 (format codec), quant (block quantisation), route (affinity,
group-limited selection, gates), permute (histogram and stable grouping
by expert), ffn (scaled FP8 contraction, SwiGLU expert), layer (whole
forward, combine, bias update), balance (sequence-wise balance loss),
backward (the layer's gradients with the expert choice held fixed, FP8
data and weight gradients, and the flags of quantised elements near an
E4M3 rounding midpoint).

Parity status: every function is pinned by tests under tests/ (closed
forms, exhaustive format checks, brute force on tiny inputs, library
special cases; the backward's gradients against finite differences). The
pages give no error bound or worked example for the layer output itself, so
the output tolerance is the one stated for the layer, not a number from the
pages; the gradients' tolerances are derived from the arithmetic.
"""
