"""Pins of the backward oracle (oracle/backward.py).

* With quantisation off, every gradient (dx, the expert weights, the router
  weight) equals central finite differences of a float64 layer written out
  here token by token, with the expert choice held fixed.
* The 128x1 grouped quantisation: padding, scale of every tile from an
  explicit loop, the amax element on +-448, the E4M3 half-spacing error bound.
* The weight-gradient contraction: exact integer products with unit scales,
  and the dense float64 product of the dequantised operands in general.
* Gate gradient: rescaling every affinity leaves the gates unchanged, so the
  affinity gradient is orthogonal to s; with quantisation on, the gradients
  stay near the exact ones.
"""
import numpy as np
import pytest

from oracle import e4m3
from oracle.bounds import CHUNK_ROUNDINGS, U
from oracle.backward import (Quantiser, dequant_128x1_grouped, gate_grad, gemm_bound, gemm_fp8_wgrad,
                             layer_backward, quant_128x1_grouped, segment_starts, swiglu_grad)


class _Cfg:
    def __init__(self, T, d, E, I, K):
        self.T, self.d, self.E, self.I, self.K = T, d, E, I, K


def _small_layer(seed=0, T=7, d=6, E=4, I=5, K=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    dy = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) / np.sqrt(d)
    W = {e: (rng.standard_normal((I, d)) / np.sqrt(d), rng.standard_normal((I, d)) / np.sqrt(d),
             rng.standard_normal((d, I)) / np.sqrt(I)) for e in range(E + 1)}
    # a fixed choice of K distinct experts per token
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    return _Cfg(T, d, E, I, K), x, dy, Wr, W, idx


def _loss(cfg, x, dy, Wr, W, idx):
    """sum_t dy[t] . y[t], y[t] = shared(x_t) + sum_k g_k FFN_{e_k}(x_t), written out per token."""
    total = 0.0
    for t in range(cfg.T):
        def ffn(e):
            w1, w3, w2 = W[e]
            a = w1 @ x[t]
            b = w3 @ x[t]
            return w2 @ (a / (1.0 + np.exp(-a)) * b)
        s = [1.0 / (1.0 + np.exp(-(x[t] @ Wr[e]))) for e in idx[t]]
        y = ffn(cfg.E)
        for k, e in enumerate(idx[t]):
            y = y + s[k] / sum(s) * ffn(e)
        total += dy[t] @ y
    return total


def _fd(f, arr, h=1e-6):
    g = np.zeros_like(arr)
    for i in np.ndindex(arr.shape):
        old = arr[i]
        arr[i] = old + h
        up = f()
        arr[i] = old - h
        dn = f()
        arr[i] = old
        g[i] = (up - dn) / (2 * h)
    return g


def test_exact_gradients_match_finite_differences():
    cfg, x, dy, Wr, W, idx = _small_layer()
    s = 1.0 / (1.0 + np.exp(-(x @ Wr.T)))
    s_sel = np.take_along_axis(s, idx, axis=1)
    Q = Quantiser(on=False)
    r = layer_backward(cfg, x, dy, Wr, idx, s_sel, lambda e: W[e], tokens=range(cfg.T),
                       wgrad_experts=range(cfg.E + 1), router_experts=range(cfg.E), Q=Q, xd=x)
    f = lambda: _loss(cfg, x, dy, Wr, W, idx)  # noqa: E731
    np.testing.assert_allclose(r["dx"], _fd(f, x), rtol=1e-6, atol=1e-7)
    dWr = _fd(f, Wr)
    for e in range(cfg.E):
        np.testing.assert_allclose(r["dWr"][e], dWr[e], rtol=1e-6, atol=1e-7)
    for e in range(cfg.E + 1):
        for j, name in enumerate(("W1", "W3", "W2")):
            np.testing.assert_allclose(r["dW"][e][j], _fd(f, W[e][j]), rtol=1e-6, atol=1e-7, err_msg=f"{name}[{e}]")
        assert not r["dW"][e][3]["dW1"].any()              # nothing is flagged without quantisation


def test_swiglu_grad_finite_differences():
    rng = np.random.default_rng(1)
    a, b, dh = rng.standard_normal((3, 50)) * 3
    h = 1e-6
    f = lambda a_, b_: (a_ / (1 + np.exp(-a_))) * b_ * dh  # noqa: E731
    dA, dB = swiglu_grad(a, b, dh)
    np.testing.assert_allclose(dA, (f(a + h, b) - f(a - h, b)) / (2 * h), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dB, (f(a, b + h) - f(a, b - h)) / (2 * h), rtol=1e-6, atol=1e-8)


def test_gate_grad_orthogonal_to_affinity():
    rng = np.random.default_rng(2)
    s = rng.uniform(0.05, 0.95, (20, 6))
    dg = rng.standard_normal((20, 6))
    dz = gate_grad(s, dg)
    ds = dz / (s * (1 - s))
    np.testing.assert_allclose((ds * s).sum(axis=1), 0.0, atol=1e-12)


@pytest.mark.parametrize("rule", ["fp32", "pow2"])
def test_quant_128x1_grouped_tiles(rule):
    rng = np.random.default_rng(3)
    sizes = [0, 5, 130, 128, 1, 0, 257]
    offsets = np.concatenate([[0], np.cumsum(sizes)])
    R, C = int(offsets[-1]), 9
    v = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-4, 4, (R, C)))).astype(np.float32)
    v[6:10, 2] = 0.0                      # a partly zero column
    v[135:263, 4] = 0.0                   # an all-zero tile (group 3, channel 4)
    qT, sT = quant_128x1_grouped(v, offsets, rule)
    P = segment_starts(offsets)
    assert list(P) == [0, 0, 128, 384, 512, 640, 640, 1024]
    assert qT.shape == (C, 1024) and sT.shape == (8, C)
    deq = dequant_128x1_grouped(qT, sT)
    for g in range(len(sizes)):
        m = sizes[g]
        for c in range(C):
            col = qT[c, P[g]:P[g + 1]]
            assert not col[m:].any(), "padding codes must be 0x00"
            for ch in range((m + 127) // 128):
                lo, hi = ch * 128, min(m, ch * 128 + 128)
                vals = [float(v[offsets[g] + i, c]) for i in range(lo, hi)]
                amax = max(abs(t) for t in vals)
                sc = float(sT[P[g] // 128 + ch, c])
                if amax == 0.0:
                    assert sc == 0.0
                    continue
                if rule == "fp32":
                    assert sc == float(np.float32(amax) / np.float32(448.0))
                    top = int(np.argmax([abs(t) for t in vals]))
                    assert col[lo + top] & 0x7F == 0x7E          # +-448
                else:
                    assert sc >= amax / 448.0 and sc / 2 < amax / 448.0 or sc == 2.0 ** -126
                    assert np.frexp(sc)[0] == 0.5
                for i in range(lo, hi):
                    t = vals[i - lo]
                    r = abs(t) / sc
                    spacing = 2.0 ** (max(np.floor(np.log2(r)), -6) - 3) if r > 0 else 2.0 ** -9
                    assert abs(deq[c, P[g] + i] - t) <= 0.5 * spacing * sc * (1 + 1e-12)


def test_wgrad_contraction_integer_exact():
    rng = np.random.default_rng(4)
    M, N, Rp = 3, 5, 256
    # small integers are exact E4M3 values; scales 1 -> a plain integer matmul
    ia = rng.integers(-8, 9, (M, Rp))
    ib = rng.integers(-8, 9, (N, Rp))
    code = {int(v): int(e4m3.encode(np.float32(v))) for v in range(-8, 9)}
    qa = np.vectorize(code.get)(ia).astype(np.uint8)
    qb = np.vectorize(code.get)(ib).astype(np.uint8)
    ones_a = np.ones((Rp // 128, M), np.float32)
    ones_b = np.ones((Rp // 128, N), np.float32)
    got = gemm_fp8_wgrad(qa, ones_a, qb, ones_b)
    want = [[sum(int(ia[m, r]) * int(ib[n, r]) for r in range(Rp)) for n in range(N)] for m in range(M)]
    assert np.array_equal(got, np.array(want, np.float64))
    # with scales: the dense product of the dequantised operands
    sa = rng.uniform(0.1, 2, (Rp // 128, M)).astype(np.float32)
    sb = rng.uniform(0.1, 2, (Rp // 128, N)).astype(np.float32)
    got = gemm_fp8_wgrad(qa, sa, qb, sb)
    A = ia * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    B = ib * np.repeat(sb.T.astype(np.float64), 128, axis=1)
    want = np.array([[sum(A[m, r] * B[n, r] for r in range(Rp)) for n in range(N)] for m in range(M)])
    np.testing.assert_allclose(got, want, rtol=1e-13)


def test_quantised_gradients_near_exact():
    """FP8 quantisation points perturb the gradients by a few per cent at most."""
    rng = np.random.default_rng(5)
    T, d, E, I, K = 40, 256, 4, 128, 2
    cfg = _Cfg(T, d, E, I, K)
    x = rng.standard_normal((T, d)).astype(np.float32)
    dy = rng.standard_normal((T, d)).astype(np.float32)
    Wr = rng.standard_normal((E, d)) / np.sqrt(d)
    W = {e: tuple(rng.standard_normal(sh) / np.sqrt(d) for sh in ((I, d), (I, d), (d, I))) for e in range(E + 1)}
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    s_sel = np.take_along_axis(1.0 / (1.0 + np.exp(-(x.astype(np.float64) @ Wr.T))), idx, axis=1)
    kw = dict(tokens=range(T), wgrad_experts=range(E + 1), router_experts=range(E))
    exact = layer_backward(cfg, x, dy, Wr, idx, s_sel, lambda e: W[e], Q=Quantiser(on=False), xd=x, **kw)
    quant = layer_backward(cfg, x, dy, Wr, idx, s_sel, lambda e: W[e], Q=Quantiser(), **kw)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)  # noqa: E731
    assert rel(quant["dx"], exact["dx"]) < 0.08
    for e in range(E + 1):
        for j in range(3):
            assert rel(quant["dW"][e][j], exact["dW"][e][j]) < 0.08


def test_quantiser_range_at_and_away_from_rounding_midpoints():
    """The range of dequantised values under an input error bound: zero for zero error; one
    whole code step for a value on a rounding midpoint of the E4M3 grid (the neighbouring codes
    are both reachable); only the scale's own relative variation for a value far from every
    boundary. In a tile whose amax is 448 * 1 (scale 1), 1.0625 sits between codes 1 and
    1.125, 0.53125 between 0.5 and 0.5625, 2^-10 on the subnormal grid (spacing 2^-9)."""
    Q = Quantiser("fp32")
    row = np.zeros((1, 128), np.float32)
    row[0, 0] = 448.0                                   # amax 448: scale exactly 1
    vals = [1.0625, 0.53125, 2.0 ** -10, 1.0, 40.0]
    row[0, 1:1 + len(vals)] = vals
    Q.rows(row, 0.0)
    assert not Q.delta.any()
    err = np.zeros((1, 128))
    err[0, 1:1 + len(vals)] = 1e-6
    Q.rows(row, err)
    d = Q.delta[0, 1:1 + len(vals)]
    assert d[0] == 0.125 and d[1] == 0.0625 and d[2] == 2.0 ** -9     # both neighbours reachable
    assert d[3] == 0.0 and d[4] == 0.0                                 # exact grid points, amax certain
    # the amax's own error moves the scale: every value then ranges with it (relative ~ err/amax)
    err[0, 0] = 448 * 1e-4
    Q.rows(row, err)
    assert 0 < Q.delta[0, 4] < 40.0 * 3e-4


def test_gemm_bound_covers_float32_chunked_evaluation():
    """gemm_bound against FP32 evaluations written out the way a chunk-promoted GEMM works:
    each 128-element chunk summed in four FP32 steps of 32 exact products (in two different
    orders), then promoted into an FP32 running sum. Every result lies within the bound of
    the exact product; the bound is not vacuous (more than 1% of it is used somewhere);
    and it is the stated formula."""
    rng = np.random.default_rng(8)
    m, k, n = 16, 1024, 24
    A = (rng.standard_normal((m, k)) * np.exp(rng.uniform(-3, 3, (m, k)))).astype(np.float32).astype(np.float64)
    B = rng.standard_normal((k, n)).astype(np.float32).astype(np.float64)
    exact = A @ B
    bound = gemm_bound(A, B)
    used = 0.0
    for order in (1, -1):
        acc = np.zeros((m, n), np.float32)
        for c in range(k // 128):
            part = np.zeros((m, n), np.float32)
            for step in range(4)[::order]:
                cols = slice(c * 128 + 32 * step, c * 128 + 32 * step + 32)
                part = (part + (A[:, cols] @ B[cols]).astype(np.float32)).astype(np.float32)
            acc = (acc + part).astype(np.float32)
        err = np.abs(acc.astype(np.float64) - exact)
        assert (err <= bound).all()
        used = max(used, float((err / bound).max()))
    assert used > 0.01
    run = np.zeros((m, n))
    acc = np.zeros((m, n))
    for c in range(0, k, 128):
        p = A[:, c:c + 128] @ B[c:c + 128]
        acc += p
        run += np.abs(p) + np.abs(acc)
    assert np.allclose(bound, U * (CHUNK_ROUNDINGS * (np.abs(A) @ np.abs(B)) + run))


def _planted_case(plant):
    """Weight gradients of a small layer, with one 128x1 code of dA moved by a step when
    `plant`, on an element whose range is far below a code step (only its tile scale may vary:
    no correct evaluation could change its code)."""
    import oracle.backward as bw
    rng = np.random.default_rng(9)
    T, d, E, I, K = 64, 256, 2, 128, 1
    cfg = _Cfg(T, d, E, I, K)
    x = rng.standard_normal((T, d)).astype(np.float32)
    dy = rng.standard_normal((T, d)).astype(np.float32)
    Wr = rng.standard_normal((E, d)) / np.sqrt(d)
    W = {e: tuple(rng.standard_normal(sh) / np.sqrt(d) for sh in ((I, d), (I, d), (d, I))) for e in range(E + 1)}
    idx = np.zeros((T, K), np.int32)
    s_sel = np.full((T, K), 0.5)
    real_tokens = bw.Quantiser.tokens
    picked = {}

    def tokens(self, v, err=0.0):
        out = real_tokens(self, v, err)
        if plant and v.shape == (T, I) and "done" not in picked:
            certain = np.argwhere((self.delta < 1e-3 * np.abs(out)) & (np.abs(out) > 0))
            t, i = certain[len(certain) // 2]
            picked.update(done=True, at=(t, i))
            out = out.copy()
            out[t, i] *= 1.0625 if abs(out[t, i]) < 0.5 * np.abs(out[:, i]).max() else 0.9375
        return out

    bw.Quantiser.tokens = tokens
    try:
        r = layer_backward(cfg, x, dy, Wr, idx, s_sel, lambda e: W[e], wgrad_experts=[0], Q=Quantiser())
    finally:
        bw.Quantiser.tokens = real_tokens
    return r["dW"][0]


def test_budget_check_catches_a_flip_outside_the_ranges():
    """The weight-gradient check a device result must meet, element by element: within
    budget + base (the quantisation ranges' effect plus the contraction's own FP32 bound) of
    the oracle. The oracle's own result passes it; the same computation with one dA code
    moved by a step, on an element whose range is only its scale's variation (no correct
    evaluation could change that code), fails it."""
    clean = _planted_case(False)
    bad = _planted_case(True)
    dW1 = clean[0]
    allow = clean[3]["dW1"] + clean[3]["base"]["dW1"]
    assert (np.abs(clean[0] - dW1) <= allow).all()
    assert (np.abs(bad[0] - dW1) > allow).any()
    # the allowance is a small part of the gradient as a whole (it cannot hide a systematic
    # error); a single row may carry more where an uncertain code sits at its column's maximum
    assert np.linalg.norm(allow) <= 2e-2 * np.linalg.norm(dW1)


def test_scaled_rows_reduces_to_plain_quantisation():
    """g * y with g = 1 or a power of two is quantised exactly like the plain 1x128 rule."""
    from oracle.quant import dequant_1x128, quant_1x128
    rng = np.random.default_rng(6)
    y = rng.standard_normal((9, 256)).astype(np.float32)
    for rule in ("fp32", "pow2"):
        Q = Quantiser(rule)
        for g in (1.0, 0.25, 2.0 ** -7):
            got = Q.scaled_rows(y, np.full(9, g))
            want = dequant_1x128(*quant_1x128((g * y).astype(np.float32), rule))
            assert np.array_equal(got, want), (rule, g)
    # a general gate: within one E4M3 step of g * y, the scale g times the plain scale
    g = rng.uniform(0.05, 0.9, 9)
    got = Quantiser("fp32").scaled_rows(y, g)
    q, s = quant_1x128(y, "fp32")
    np.testing.assert_allclose(got, dequant_1x128(q, s) * g[:, None], rtol=2 ** -23)
