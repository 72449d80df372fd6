"""Pins for the whole oracle layer: a per-token scalar brute force on tiny
inputs, the all-experts special case, token independence and the residual."""
import itertools
import math

import numpy as np
import pytest

from oracle.layer import Layer
from oracle.quant import dequant_128x128, dequant_1x128, quant_1x128
from sparse_moe_layer_13_b300.configs import MoEConfig
from sparse_moe_layer_13_b300 import inputs

CFG = MoEConfig("pin", T=6, d=256, E=8, I=128, K=3, G=4, M=2, gk=2, seed=11, bias="uniform")


def _make(cfg):
    x = inputs.gen_x(cfg).float().numpy()
    Wr = inputs.gen_router(cfg).numpy()
    b = inputs.gen_bias(cfg).numpy()
    wts = {e: [w.numpy() for w in inputs.gen_expert(cfg, e)] for e in range(cfg.E + 1)}
    return x, Wr, b, wts


def _brute_token(cfg, x, Wr, b, layer, t, rule="fp32"):
    s = [1 / (1 + math.exp(-math.fsum(x[t, j] * Wr[e, j] for j in range(cfg.d)))) for e in range(cfg.E)]
    sb = [s[e] + float(b[e]) for e in range(cfg.E)]
    n = cfg.E // cfg.G
    score = [sum(sorted(sb[g * n:(g + 1) * n], reverse=True)[:cfg.gk]) for g in range(cfg.G)]
    groups = max(itertools.combinations(range(cfg.G), cfg.M), key=lambda c: sum(score[g] for g in c))
    cand = [e for g in groups for e in range(g * n, (g + 1) * n)]
    chosen = max(itertools.combinations(cand, cfg.K), key=lambda c: sum(sb[e] for e in c))
    tot = sum(s[e] for e in chosen)
    xq, xs = quant_1x128(x[t:t + 1], rule)
    X = dequant_1x128(xq, xs)[0]

    def ffn(e):
        ex = layer.expert(e)
        W1, W3, W2 = (dequant_128x128(ex.q1, ex.s1), dequant_128x128(ex.q3, ex.s3), dequant_128x128(ex.q2, ex.s2))
        h = np.array([np.float32((lambda g, u: g / (1 + math.exp(-g)) * u)(
            math.fsum(X * W1[j]), math.fsum(X * W3[j]))) for j in range(cfg.I)], np.float32)
        hq, hs = quant_1x128(h[None, :], rule)
        H = dequant_1x128(hq, hs)[0]
        return np.array([math.fsum(H * W2[i]) for i in range(cfg.d)])

    y = ffn(cfg.E)
    for e in chosen:
        y = y + (s[e] / tot) * ffn(e)
    return set(chosen), y


def test_layer_matches_scalar_brute_force():
    x, Wr, b, wts = _make(CFG)
    layer = Layer(CFG, Wr, b, lambda e: wts[e])
    res = layer.forward(x)
    for t in range(CFG.T):
        chosen, y = _brute_token(CFG, x, Wr, b, layer, t)
        assert set(res["idx"][t]) == chosen
        # the two sums of h may round to float32 differently in the last place
        assert np.max(np.abs(res["y"][t] - y)) <= 1e-6 * np.max(np.abs(y))


def test_layer_pow2_rule_matches_scalar_brute_force():
    """The power-of-two scale rule flows through every quantisation of the layer
    (x, the weights and h): the layer equals the scalar evaluation with that rule."""
    x, Wr, b, wts = _make(CFG)
    layer = Layer(CFG, Wr, b, lambda e: wts[e], rule="pow2")
    res = layer.forward(x)
    for e in range(CFG.E + 1):
        ex = layer.expert(e)
        for sc in (ex.s1, ex.s3, ex.s2):
            assert np.all(np.frexp(sc.astype(np.float64))[0] == 0.5)
    for t in range(CFG.T):
        chosen, y = _brute_token(CFG, x, Wr, b, layer, t, rule="pow2")
        assert set(res["idx"][t]) == chosen
        assert np.max(np.abs(res["y"][t] - y)) <= 1e-6 * np.max(np.abs(y))
    ref = Layer(CFG, Wr, b, lambda e: wts[e]).forward(x)["y"]
    assert not np.array_equal(res["y"], ref)      # a different quantisation rule gives different bytes


def test_all_experts_special_case():
    cfg = MoEConfig("all", T=5, d=128, E=4, I=128, K=4, G=2, M=2, gk=1, seed=12)
    x, Wr, b, wts = _make(cfg)
    layer = Layer(cfg, Wr, b, lambda e: wts[e])
    res = layer.forward(x)
    s = 1 / (1 + np.exp(-(x.astype(np.float64) @ Wr.astype(np.float64).T)))
    g = s / s.sum(1, keepdims=True)
    xq, xs = quant_1x128(x)
    from oracle.ffn import expert_forward
    y = expert_forward(xq, xs, layer.expert(4))
    for e in range(4):
        y = y + g[:, e:e + 1] * expert_forward(xq, xs, layer.expert(e))
    np.testing.assert_allclose(res["y"], y, rtol=1e-12, atol=1e-12)


def test_tokens_are_independent_and_subset_matches():
    x, Wr, b, wts = _make(CFG)
    layer = Layer(CFG, Wr, b, lambda e: wts[e])
    full = layer.forward(x)["y"]
    perm = np.array([3, 0, 5, 1, 4, 2])
    pr = layer.forward(x[perm])["y"]
    assert np.array_equal(pr, full[perm])
    sub = layer.forward(x, tokens=np.array([4, 1]))["y"]
    assert np.array_equal(sub, full[[4, 1]])


def test_residual_adds_input():
    x, Wr, b, wts = _make(CFG)
    layer = Layer(CFG, Wr, b, lambda e: wts[e])
    y0 = layer.forward(x)["y"]
    y1 = layer.forward(x, residual=True)["y"]
    np.testing.assert_allclose(y1, y0 + x, rtol=1e-12, atol=1e-12)


def test_forward_budget_covers_perturbed_evaluations():
    """Another correct evaluation of an expert, simulated: the gate and up GEMM outputs moved
    to the corners of their error bounds (bounds.gemm_bound), h recomputed and requantised
    1x128, the down projection applied. Its output lies within expert_forward's budget of the
    oracle's, element by element, for many random perturbations, and some perturbation really
    changes h codes (the budget is not vacuous)."""
    from oracle.ffn import QuantExpert, expert_forward, gemm_fp8, silu
    from oracle.quant import quant_1x128
    rng = np.random.default_rng(21)
    m, d, I = 24, 512, 256
    x = rng.standard_normal((m, d)).astype(np.float32)
    w = QuantExpert(*(rng.standard_normal(sh).astype(np.float32) / np.sqrt(d) for sh in ((I, d), (I, d), (d, I))))
    xq, xs = quant_1x128(x)
    out, budget = expert_forward(xq, xs, w, budget=True)
    gate, eg = gemm_fp8(xq, xs, w.q1, w.s1, with_bound=True)
    up, eu = gemm_fp8(xq, xs, w.q3, w.s3, with_bound=True)
    hq0, _ = quant_1x128((silu(gate) * up).astype(np.float32))
    changed = 0
    for trial in range(40):
        # extreme points of the error boxes make code changes likely near boundaries
        gp = gate + eg * rng.choice([-1.0, 1.0], gate.shape)
        upp = up + eu * rng.choice([-1.0, 1.0], up.shape)
        h = (silu(gp) * upp).astype(np.float32)
        hq, hs = quant_1x128(h)
        changed += int((hq != hq0).sum())
        o = gemm_fp8(hq, hs, w.q2, w.s2)
        assert (np.abs(o - out) <= budget * (1 + 1e-9) + 1e-12).all(), trial
    assert changed > 0
