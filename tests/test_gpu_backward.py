"""GPU parity of the backward pass against the FP64 oracle (oracle/backward.py).

Kernel by kernel on seeded synthetic operands (bit-exact for E4M3 codes,
scales and transposed bytes; FP32 tolerances for sums), then the whole
layer backward on the workload shapes: every gradient at tiny size, sampled
tokens and experts at mid and full width.

The layer gradients are held to bounds derived from the arithmetic
(oracle/bounds.py), with no tolerance of their own. The gradient GEMMs
requantise FP32 values (h, dO, dA, dB) to E4M3, and those values differ
between two correct evaluations by at most their error bounds (the producing
GEMMs' (nkc + 10) * 2^-24 * sum|terms|, carried through SiLU and its gradient,
and the gates' bound); where that interval spans an E4M3 rounding boundary
either code is correct. The oracle turns the intervals into a budget per
gradient element (how far the rounding decisions alone can move it).
  * dx, dz, dg, dWr (through bf16 rows and the layer's FP32 sums): the
    forward's bars, relative L2 <= 5e-3 of the whole difference and max |diff|
    <= 2e-2 * RMS of what the budget does not explain.
  * dW1, dW3, dW2 (FP32 contractions over tokens): element by element within
    budget + the contraction's own gemm_bound.
  * every budget at most 5% of its gradient as a whole (gpu_helpers.BUDGET_CAP), except
    dWr's: a sum of dz x over every token of an expert, whose budget adds the tokens'
    without the cancellation the sum has (about 12% at mid width), held by the raw bars.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (BUDGET_CAP, assert_y_close, check_routing, gpu, oracle_experts, require_gpu, to_np,
                         y_metrics)
from oracle import e4m3
from oracle.backward import (Quantiser, dequant_128x1_grouped, dequant_expert, gemm_fp8_wgrad, layer_backward,
                             quant_128x1_grouped, segment_starts, swiglu_grad)
from oracle.bounds import gemm_bound
from oracle.quant import quant_1x128
from oracle.route import affinity, route as oracle_route
from sparse_moe_layer_13_b300.configs import CONFIGS

SIZES = [0, 5, 130, 128, 1, 0, 257, 384]


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _codes(rng, shape):
    """Seeded finite E4M3 codes (no NaN)."""
    c = rng.integers(0, 256, shape).astype(np.uint8)
    return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def _check_q1(B, offs, qT, sT, want_q, want_s):
    P = segment_starts(offs)
    width = int(P[-1])
    assert np.array_equal(to_np(qT)[:, :width], want_q), "128x1 codes differ"
    got_s = to_np(sT)[:width // 128]
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), "128x1 scales differ"


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_quant_128x1_f32_source(rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(10)
    offs = _offsets(SIZES)
    R, C = int(offs[-1]) + 3, 384                      # three trailing rows outside every group
    v = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-6, 6, (R, C)))).astype(np.float32)
    v[7:20, 5] = 0.0
    qT, sT = B.quant_128x1(torch.from_numpy(offs).cuda(), R, C, rule, f32=torch.from_numpy(v).cuda())
    want_q, want_s = quant_128x1_grouped(v, offs, rule)
    _check_q1(B, offs, qT, sT, want_q, want_s)


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_quant_128x1_fp8_source(rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(11)
    offs = _offsets(SIZES)
    R, C = int(offs[-1]), 256
    q = _codes(rng, (R, C))
    s = rng.uniform(1e-3, 4.0, (R, C // 128)).astype(np.float32)
    qT, sT = B.quant_128x1(torch.from_numpy(offs).cuda(), R, C, rule,
                           fp8=(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()))
    vals = (e4m3.decode(q).reshape(R, C // 128, 128) * s.astype(np.float64)[:, :, None]).reshape(R, C)
    want_q, want_s = quant_128x1_grouped(vals.astype(np.float32), offs, rule)
    _check_q1(B, offs, qT, sT, want_q, want_s)


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_quant_128x1_bf16_rows_source(rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(12)
    offs = _offsets(SIZES)
    R, C, X = int(offs[-1]), 256, 300
    x = _bf16(rng.standard_normal((X, C)) * 3)
    row_map = rng.integers(0, X, R).astype(np.int32)
    mult = rng.uniform(0.01, 1.0, R).astype(np.float32)
    qT, sT = B.quant_128x1(torch.from_numpy(offs).cuda(), R, C, rule,
                           bf16_rows=(x.cuda(), torch.from_numpy(row_map).cuda(), torch.from_numpy(mult).cuda()))
    xf = x.float().numpy().astype(np.float64)
    vals = (mult.astype(np.float64)[:, None] * xf[row_map]).astype(np.float32)
    want_q, want_s = quant_128x1_grouped(vals, offs, rule)
    _check_q1(B, offs, qT, sT, want_q, want_s)


@gpu
def test_transpose_fp8_blocks():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(13)
    b, rows, cols = 3, 256, 384
    q = _codes(rng, (b, rows, cols))
    s = rng.uniform(0.1, 2, (b, rows // 128, cols // 128)).astype(np.float32)
    qT, sT = B.transpose_fp8_blocks(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    assert np.array_equal(to_np(qT), q.transpose(0, 2, 1))
    assert np.array_equal(to_np(sT), s.transpose(0, 2, 1))
    # two matrices side by side, padded rows left alone
    wide = torch.full((b, cols + 128, 2 * rows), 7, dtype=torch.uint8, device="cuda")
    wide_s = torch.full((b, (cols + 128) // 128, 2 * rows // 128), -1.0, device="cuda")
    B.transpose_fp8_blocks(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), wide, wide_s, offset=rows)
    w = to_np(wide)
    assert np.array_equal(w[:, :cols, rows:], q.transpose(0, 2, 1))
    assert (w[:, :cols, :rows] == 7).all() and (w[:, cols:] == 7).all()
    assert np.array_equal(to_np(wide_s)[:, :cols // 128, rows // 128:], s.transpose(0, 2, 1))


@gpu
@pytest.mark.parametrize("sizes", [SIZES, [0, 0, 1], [1024, 64, 0, 640]])
def test_grouped_wgrad_fp8(sizes):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(14)
    offs = _offsets(sizes)
    G = len(sizes)
    P = segment_starts(offs)
    M, N = 256, 512
    width = B.q1_width(G, int(offs[-1]))
    aT = np.zeros((M, width), np.uint8)
    bT = np.zeros((N, width), np.uint8)
    aT[:, :P[-1]] = _codes(rng, (M, int(P[-1])))
    bT[:, :P[-1]] = _codes(rng, (N, int(P[-1])))
    saT = rng.uniform(1e-3, 1e-2, (width // 128, M)).astype(np.float32)
    sbT = rng.uniform(1e-3, 1e-2, (width // 128, N)).astype(np.float32)
    out = B.grouped_wgrad_fp8(torch.from_numpy(offs).cuda(), int(offs[-1]), torch.from_numpy(aT).cuda(),
                              torch.from_numpy(saT).cuda(), torch.from_numpy(bT).cuda(), torch.from_numpy(sbT).cuda())
    B.check_device_status()
    got = to_np(out)
    for g in range(G):
        c0, c1 = int(P[g]), int(P[g + 1])
        if c1 == c0:
            assert not got[g].any(), f"group {g} has no rows but a nonzero gradient"
            continue
        want = gemm_fp8_wgrad(aT[:, c0:c1], saT[c0 // 128:c1 // 128], bT[:, c0:c1], sbT[c0 // 128:c1 // 128])
        rel = np.linalg.norm(got[g] - want) / np.linalg.norm(want)
        assert rel < 1e-5, f"group {g}: rel-L2 {rel:.3e}"
        # element by element within the evaluation bound of the oracle's budgets (oracle/bounds.py)
        Ad = dequant_128x1_grouped(aT[:, c0:c1], saT[c0 // 128:c1 // 128])
        Bd = dequant_128x1_grouped(bT[:, c0:c1], sbT[c0 // 128:c1 // 128])
        bound = gemm_bound(Ad, Bd.T)
        assert (np.abs(got[g] - want) <= bound).all(), f"group {g}: beyond the evaluation bound"


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_swiglu_backward(rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding as B
    rng = np.random.default_rng(15)
    rows, I = 200, 384
    a = (rng.standard_normal((rows, I)) * 3).astype(np.float32)
    b = (rng.standard_normal((rows, I)) * 2).astype(np.float32)
    dh = rng.standard_normal((rows, I + 128)).astype(np.float32)
    # gate/up tile layout: I-block j -> gate[128j..+64) up[..] gate[128j+64..+128) up[..]
    ab = np.empty((rows, 2 * I), np.float32)
    for j in range(I // 128):
        for h in range(2):
            sl = slice(128 * j + 64 * h, 128 * j + 64 * h + 64)
            ab[:, 256 * j + 128 * h: 256 * j + 128 * h + 64] = a[:, sl]
            ab[:, 256 * j + 128 * h + 64: 256 * j + 128 * h + 128] = b[:, sl]
    abt = torch.from_numpy(ab).cuda()
    q = torch.empty(rows, 2 * I, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, 2 * I // 128, dtype=torch.float32, device="cuda")
    B.swiglu_backward(abt, torch.from_numpy(dh).cuda(), q, s, rule)
    dA, dB = swiglu_grad(a, b, dh[:, :I])
    out = to_np(abt)
    got_a = np.empty_like(a)
    got_b = np.empty_like(b)
    for j in range(I // 128):
        for h in range(2):
            sl = slice(128 * j + 64 * h, 128 * j + 64 * h + 64)
            got_a[:, sl] = out[:, 256 * j + 128 * h: 256 * j + 128 * h + 64]
            got_b[:, sl] = out[:, 256 * j + 128 * h + 64: 256 * j + 128 * h + 128]
    for got, want in ((got_a, dA), (got_b, dB)):
        err = np.abs(got - want) / (np.abs(want).max(axis=1, keepdims=True) + 1e-30)
        assert err.max() < 1e-5
    # 1x128 E4M3 of [dA | dB]: the oracle quantises its own float32 rounding of the exact values,
    # so an element whose two roundings straddle an E4M3 rounding boundary may differ by one code
    wq, ws = quant_1x128(np.concatenate([dA, dB], axis=1).astype(np.float32), rule)
    gq, gs = to_np(q), to_np(s)
    np.testing.assert_allclose(gs, ws, rtol=1e-5)
    same = gq == wq
    assert same.mean() > 0.999
    dq = e4m3.decode(gq[~same]).astype(np.float64)
    dw = e4m3.decode(wq[~same]).astype(np.float64)
    assert (np.abs(dq - dw) <= np.abs(dw) * 0.125 + 2.0 ** -9).all()


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_combine_backward(rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    from sparse_moe_layer_13_b300.configs import MoEConfig
    cfg = MoEConfig("t", T=96, d=384, E=16, I=128, K=4, G=4, M=2, gk=2, seed=0)
    rng = np.random.default_rng(16)
    T, K, d = cfg.T, cfg.K, cfg.d
    dy = _bf16(rng.standard_normal((T, d)))
    routed = _bf16(rng.standard_normal((T * K, d)))
    row_of = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    gate = rng.uniform(0.01, 0.7, (T, K)).astype(np.float32)
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    dOq = torch.empty(cfg.rows, d, dtype=torch.uint8, device="cuda")
    dOs = torch.empty(cfg.rows, d // 128, dtype=torch.float32, device="cuda")
    rgate = torch.empty(cfg.rows, dtype=torch.float32, device="cuda")
    dgate = torch.empty(T, K, dtype=torch.float32, device="cuda")
    binding.combine_backward(cfg, dy.cuda(), routed.cuda(), dev(row_of), dev(gate), dOq, dOs, rgate, dgate, rule)
    binding.check_device_status()
    dyf = dy.float().numpy().astype(np.float64)
    rf = routed.float().numpy().astype(np.float64)
    want_rg = np.ones(cfg.rows, np.float32)
    rows_g = np.ones(cfg.rows)
    src = np.zeros((cfg.rows, d), np.float32)
    for t in range(T):
        for k in range(K):
            src[row_of[t, k]] = dyf[t]
            rows_g[row_of[t, k]] = gate[t, k]
            want_rg[row_of[t, k]] = gate[t, k]
        src[T * K + t] = dyf[t]
    if rule == "fp32":
        # codes of dy's own tiles, scale fl32(g * s)
        wq, s_dy = quant_1x128(src, rule)
        ws = (rows_g[:, None] * s_dy.astype(np.float64)).astype(np.float32)
    else:
        wq, ws = quant_1x128((rows_g[:, None] * src.astype(np.float64)).astype(np.float32), rule)
    assert np.array_equal(to_np(dOq), wq)
    assert np.array_equal(to_np(dOs).view(np.uint32), ws.view(np.uint32))
    assert np.array_equal(to_np(rgate), want_rg)
    want_dg = np.array([[dyf[t] @ rf[row_of[t, k]] for k in range(K)] for t in range(T)])
    np.testing.assert_allclose(to_np(dgate), want_dg, rtol=1e-4, atol=1e-4 * np.abs(want_dg).max())


# ----------------------------------------------------------------- the layer ----
def _unpack_w13(dW13_e, I):
    """Rows of a gradient in the SwiGLU tile layout -> (dW1 [I][*], dW3 [I][*])."""
    p = np.arange(2 * I)
    j, q = p // 256, p % 256
    up = ((q >= 64) & (q < 128)) | (q >= 192)
    i = 128 * j + np.where(q < 128, q % 64, 64 + q % 64)
    dW1 = np.empty((I, dW13_e.shape[1]), dW13_e.dtype)
    dW3 = np.empty_like(dW1)
    dW1[i[~up]] = dW13_e[~up]
    dW3[i[up]] = dW13_e[up]
    return dW1, dW3


def _check_wgrad(name, got, want, budget, base):
    """Element by element within budget + base; the budget a small part of the gradient."""
    allow = budget + base
    diff = np.abs(got.astype(np.float64) - want)
    over = diff > allow
    share = np.linalg.norm(budget) / np.linalg.norm(want)
    rel, mx = y_metrics(got, want)
    print(f"[parity] {name}: rel-L2 {rel:.3e} max-abs/RMS {mx:.3e}; budget {share:.2e} of the gradient; "
          f"worst |diff| / (budget + base) {np.max(diff / np.maximum(allow, 1e-300)):.3f}; "
          f"{over.sum()} of {over.size} elements beyond it")
    assert share <= BUDGET_CAP, f"{name}: budget {share:.3e} of the gradient"
    assert not over.any(), f"{name}: {over.sum()} elements beyond budget + base"


def _backward_case(cfg, tokens=None, wgrad_experts=None, router_experts=None, rule="fp32", seed=0):
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.layer import MoELayer
    layer = MoELayer(cfg, "cuda", scale_rule=rule, backward=True)
    x = inputs.gen_x(cfg, "cuda")
    dy = inputs.gen_dy(cfg, "cuda")
    b0 = to_np(layer.bias).copy()
    layer.forward(x, update_bias=False)
    g = layer.backward(x, dy)
    binding.check_device_status()
    xn, Wr, dyn = to_np(x), to_np(layer.Wr), to_np(dy)
    ref_idx, ref_gate, info = oracle_route(xn, Wr, b0, cfg.G, cfg.M, cfg.K, cfg.gk)
    gidx = to_np(layer.idx)
    tie, _ = check_routing(cfg, gidx, to_np(layer.gate), ref_idx, ref_gate, info)
    s_sel = np.take_along_axis(affinity(xn, Wr), ref_idx, axis=1)
    rng = np.random.default_rng(seed)
    ok_tok = np.nonzero(~tie)[0]
    tokens = ok_tok if tokens is None else np.sort(rng.choice(ok_tok, tokens, replace=False))
    # an expert's weight gradient sums over its rows: only experts no near-tie token reaches
    tied = set(ref_idx[tie].ravel().tolist()) | set(gidx[tie].ravel().tolist())
    wgrad_experts = [e for e in (range(cfg.E + 1) if wgrad_experts is None else wgrad_experts) if e not in tied]
    router_experts = [e for e in (range(cfg.E) if router_experts is None else router_experts) if e not in tied]
    need = set(ref_idx[tokens].ravel().tolist()) | {cfg.E} | set(wgrad_experts)
    for e in router_experts:
        for t in np.nonzero((ref_idx == e).any(axis=1))[0]:
            need |= set(ref_idx[t].tolist())
    ex = oracle_experts(cfg, need, rule=rule)
    deq = {e: dequant_expert(w) for e, w in ex.items()}
    Q = Quantiser(rule)
    ref = layer_backward(cfg, xn, dyn, Wr, ref_idx, s_sel, lambda e: deq[e], tokens=tokens,
                         wgrad_experts=wgrad_experts, router_experts=router_experts, Q=Q)
    bud = ref["budget"]
    print(f"[backward {cfg.name} {rule}] {len(tokens)} tokens, experts {wgrad_experts}, router rows {router_experts}")
    assert_y_close(to_np(g["dx"])[tokens], ref["dx"], bud["dx"], name="dx")
    ti = ref_idx[tokens]
    order_g, order_r = np.argsort(gidx[tokens], axis=1), np.argsort(ti, axis=1)
    by = lambda v, o: np.take_along_axis(v, o, axis=1)  # noqa: E731
    assert_y_close(by(to_np(g["dz"])[tokens], order_g), by(ref["dz"], order_r), by(bud["dz"], order_r), name="dz")
    assert_y_close(by(to_np(g["dgate"])[tokens], order_g), by(ref["dg"], order_r), by(bud["dg"], order_r),
                   name="dgate")
    for e in wgrad_experts:
        dW1, dW3, dW2, b = ref["dW"][e]
        g1, g3 = _unpack_w13(to_np(g["dW13"][e]), cfg.I)
        g2 = to_np(g["dW2T"][e]).T
        _check_wgrad(f"dW1[{e}]", g1, dW1, b["dW1"], b["base"]["dW1"])
        _check_wgrad(f"dW3[{e}]", g3, dW3, b["dW3"], b["base"]["dW3"])
        _check_wgrad(f"dW2[{e}]", g2, dW2, b["dW2"], b["base"]["dW2"])
    if router_experts:
        got = to_np(g["dWr"])[router_experts]
        want = np.stack([ref["dWr"][e] for e in router_experts])
        # dWr sums dz x over every token of an expert: its budget grows like the square root of
        # the token count against the gradient (no cancellation), so only the raw bars hold it
        assert_y_close(got, want, np.stack([bud["dWr"][e] for e in router_experts]), name="dWr", cap=False)
    return layer


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_layer_backward_tiny(rule):
    require_gpu()
    _backward_case(CONFIGS["tiny"], rule=rule)


@gpu
def test_layer_backward_mid_sampled():
    require_gpu()
    _backward_case(CONFIGS["mid"], tokens=48, wgrad_experts=[0, 37, 64], router_experts=[5, 63])


@gpu
def test_layer_backward_full_sampled():
    require_gpu()
    _backward_case(CONFIGS["full"], tokens=12, wgrad_experts=[3, 200], router_experts=[])
