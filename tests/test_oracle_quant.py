"""Pins for the oracle's 1x128 / 128x128 quantisation (closed forms, the
hand-worked tile, error bound of round-to-nearest, block-index checks)."""
from fractions import Fraction

import numpy as np

from conftest import read_golden
from oracle import e4m3
from oracle.quant import dequant_128x128, dequant_1x128, quant_128x128, quant_1x128


def _fl32(fr: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational, via exact search."""
    f = np.float32(float(fr))  # float() is correctly rounded to float64; refine to float32 below
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.frombuffer(c.tobytes(), np.uint32)[0]) & 1))
    return np.float32(best)


def test_golden_tile():
    g = read_golden("quant_tile_example.txt")
    vals = np.zeros(128, np.float32)
    head = np.array([float(v) for v in g["values"][0]], np.float32)
    vals[:len(head)] = head
    q, s = quant_1x128(vals[None, :])
    assert s[0, 0] == np.float32(g["scale"][0][0])
    assert [int(c) for c in q[0, :len(head)]] == [int(c, 16) for c in g["codes"][0]]
    assert np.all(q[0, len(head):] == 0)


def test_scale_is_correctly_rounded_quotient():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
    q, s = quant_1x128(x)
    for r in range(0, 64, 7):
        for c in range(4):
            amax = np.abs(x[r, c * 128:(c + 1) * 128]).max()
            assert s[r, c] == _fl32(Fraction(float(amax)) / 448)


def test_amax_maps_to_448_and_error_bound():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((32, 1024)) * 3).astype(np.float32)
    q, s = quant_1x128(x)
    t = x.reshape(32, 8, 128)
    qt = q.reshape(32, 8, 128)
    am = np.abs(t).argmax(axis=2)
    for r in range(32):
        for c in range(8):
            code = int(qt[r, c, am[r, c]])
            assert code in (0x7E, 0xFE)
    # round-to-nearest: |dec(q) - v/s| <= half the E4M3 spacing at that magnitude
    r = (x.reshape(32, 8, 128) / s[:, :, None]).astype(np.float32)
    dq = e4m3.decode(q).reshape(32, 8, 128)
    a = np.abs(r.astype(np.float64))
    exp = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    spacing = 2.0 ** (exp - 3)
    assert np.all(np.abs(dq - r) <= spacing / 2 + 1e-300)


def test_zero_tile():
    x = np.zeros((2, 256), np.float32)
    x[1, :128] = -0.0
    x[1, 128] = 1.0
    q, s = quant_1x128(x)
    assert np.all(s[0] == 0) and s[1, 0] == 0 and s[1, 1] > 0
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80)


def test_block_scales_index_rows_then_cols():
    w = np.ones((256, 384), np.float32)
    for i in range(2):
        for j in range(3):
            w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] *= (i * 3 + j + 1) * 4.0
    q, s = quant_128x128(w)
    assert s.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            assert s[i, j] == np.float32((i * 3 + j + 1) * 4.0 / 448)
    assert np.all(q == 0x7E)
    assert np.allclose(dequant_128x128(q, s), w, rtol=0, atol=1e-5 * w.max())


def test_dequant_close():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 256)).astype(np.float32)
    q, s = quant_1x128(x)
    rel = np.linalg.norm(dequant_1x128(q, s) - x) / np.linalg.norm(x)
    assert rel < 0.04      # 3 mantissa bits: relative rounding error <= 2^-4 per element


# ---- power-of-two (block-scaled MX) rule -----------------------------------

def _pow2_by_search(amax: float) -> float:
    """Smallest 2^e (e >= -126) with 448 * 2^e >= amax, by walking e upwards in exact arithmetic."""
    if amax == 0:
        return 0.0
    a = Fraction(float(amax))
    e = -160
    while Fraction(448) * Fraction(2) ** e < a:
        e += 1
    return float(Fraction(2) ** max(e, -126))


def test_pow2_scale_is_smallest_power_of_two_bound():
    from oracle.quant import pow2_scale
    rng = np.random.default_rng(4)
    amax = np.concatenate([
        (rng.standard_normal(300) ** 2 * 10.0 ** rng.integers(-30, 30, 300)).astype(np.float32),
        np.float32([448.0, 447.99997, 448.00003, 1.75, 1.75 * 2 ** -20, 1.7500001, 3.5, 2.0 ** -120, 1e-40, 0.0]),
    ])
    got = pow2_scale(amax)
    for a, s in zip(amax, got):
        assert float(s) == _pow2_by_search(float(a)), (a, s)


def test_pow2_quant_exact_shift_and_range():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((24, 512)) * rng.uniform(1e-6, 1e6, (24, 1))).astype(np.float32)
    q, s = quant_1x128(x, rule="pow2")
    m, ex = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)                                   # powers of two
    t = x.reshape(24, 4, 128).astype(np.float64)
    r = t / s[:, :, None].astype(np.float64)
    assert np.all(r * s[:, :, None] == t)                     # v / s is exact
    amax = np.abs(t).max(axis=2)
    assert np.all(amax / s <= 448) and np.all(amax / s > 224)  # smallest such power
    # codes are the E4M3 rounding of the exact ratio
    assert np.array_equal(q.reshape(24, 4, 128), e4m3.encode(r.astype(np.float32)))


def test_pow2_clamp_and_zero_tiles():
    x = np.zeros((3, 256), np.float32)
    x[1, 5] = 2.0 ** -133                  # smallest bf16 subnormal: scale clamps to 2^-126
    x[2, :128] = -0.0
    q, s = quant_1x128(x, rule="pow2")
    assert s[0, 0] == 0 and s[2, 0] == 0
    assert s[1, 0] == np.float32(2.0 ** -126)
    assert e4m3.decode(q[1:2, 5:6])[0, 0] * 2.0 ** -126 == 2.0 ** -133   # 2^-7 is an E4M3 subnormal
    assert np.all(q[2, :128] == 0x80)


def test_pow2_block_scales():
    w = np.ones((256, 256), np.float32)
    w[:128, 128:] *= 3.0
    w[128:, :128] *= 1000.0
    q, s = quant_128x128(w, rule="pow2")
    assert s[0, 0] == np.float32(2.0 ** -8)      # 448 * 2^-8 = 1.75 >= 1 > 0.875
    assert s[0, 1] == np.float32(2.0 ** -7)      # 3.5 >= 3
    assert s[1, 0] == np.float32(2.0 ** 2)       # 1792 >= 1000 > 896
    assert np.allclose(dequant_128x128(q, s), w, rtol=2 ** -4, atol=0)
