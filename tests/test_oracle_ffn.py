"""Pins for the oracle's scaled FP8 contraction, SwiGLU expert and bf16
rounding: exact integer products, power-of-two chunk scales against a dense
dequantised product, closed forms, torch's bf16 cast, scalar brute force."""
import math

import numpy as np
import torch

from oracle import e4m3
from oracle.ffn import QuantExpert, expert_forward, gemm_fp8, round_bf16, silu
from oracle.quant import dequant_128x128, dequant_1x128, quant_1x128

INT_CODES = {int(v): c for c, v in enumerate(e4m3.DECODE_TABLE[:0x7F]) if float(v).is_integer() and 0 < v <= 16}


def _int_operand(rng, rows, cols):
    vals = rng.integers(-16, 17, (rows, cols))
    codes = np.zeros((rows, cols), np.uint8)
    for v, c in INT_CODES.items():
        codes[vals == v] = c
        codes[vals == -v] = c | 0x80
    return vals, codes


def test_unit_scales_give_integer_matmul():
    rng = np.random.default_rng(0)
    a, qa = _int_operand(rng, 37, 384)
    b, qb = _int_operand(rng, 256, 384)
    out = gemm_fp8(qa, np.ones((37, 3), np.float32), qb, np.ones((2, 3), np.float32))
    assert np.array_equal(out, (a.astype(np.int64) @ b.T.astype(np.int64)).astype(np.float64))


def test_chunk_scales_index_row_chunk_and_block():
    rng = np.random.default_rng(1)
    a, qa = _int_operand(rng, 20, 384)
    b, qb = _int_operand(rng, 384, 384)
    sa = np.ldexp(1.0, rng.integers(-6, 6, (20, 3))).astype(np.float32)
    sb = np.ldexp(1.0, rng.integers(-6, 6, (3, 3))).astype(np.float32)
    dense = dequant_1x128(qa, sa) @ dequant_128x128(qb, sb).T   # scale every element, then one product
    assert np.array_equal(gemm_fp8(qa, sa, qb, sb), dense)


def test_general_scales_close_to_dense():
    rng = np.random.default_rng(2)
    qa = rng.integers(0, 256, (16, 512)).astype(np.uint8)
    qb = rng.integers(0, 256, (128, 512)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0
    qb[(qb & 0x7F) == 0x7F] = 0
    sa = rng.uniform(0.01, 1, (16, 4)).astype(np.float32)
    sb = rng.uniform(0.01, 1, (1, 4)).astype(np.float32)
    dense = dequant_1x128(qa, sa) @ dequant_128x128(qb, sb).T
    np.testing.assert_allclose(gemm_fp8(qa, sa, qb, sb), dense, rtol=1e-12, atol=1e-9)


def test_silu_closed_forms():
    x = np.linspace(-20, 20, 81)
    np.testing.assert_allclose(silu(x) - silu(-x), x, rtol=0, atol=1e-12)
    assert silu(0.0) == 0.0
    np.testing.assert_allclose(silu(np.log(3.0)), np.log(3.0) * 0.75, rtol=1e-15)


def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(100_000) * 10.0 ** rng.integers(-30, 30, 100_000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(round_bf16(v.astype(np.float64)), ref)


def test_expert_matches_scalar_brute_force():
    rng = np.random.default_rng(4)
    d, I = 256, 128
    w1 = rng.standard_normal((I, d)).astype(np.float32) / 16
    w3 = rng.standard_normal((I, d)).astype(np.float32) / 16
    w2 = rng.standard_normal((d, I)).astype(np.float32) / 16
    x = rng.standard_normal((3, d)).astype(np.float32)
    xq, xs = quant_1x128(x)
    ex = QuantExpert(w1, w3, w2)
    out = expert_forward(xq, xs, ex)
    W1 = dequant_128x128(ex.q1, ex.s1)
    W3 = dequant_128x128(ex.q3, ex.s3)
    W2 = dequant_128x128(ex.q2, ex.s2)
    X = dequant_1x128(xq, xs)
    for m in range(3):
        h = np.zeros(I, np.float32)
        for j in range(I):
            g = math.fsum(X[m, k] * W1[j, k] for k in range(d))
            u = math.fsum(X[m, k] * W3[j, k] for k in range(d))
            h[j] = np.float32(g / (1 + math.exp(-g)) * u)
        hq, hs = quant_1x128(h[None, :])
        H = dequant_1x128(hq, hs)[0]
        for n in range(0, d, 17):
            o = math.fsum(H[j] * W2[n, j] for j in range(I))
            assert abs(out[m, n] - o) <= 1e-12 * abs(o) + 1e-15
