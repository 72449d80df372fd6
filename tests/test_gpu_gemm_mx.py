"""GPU parity: the block-scaled grouped FP8 GEMM (power-of-two scales applied
by tcgen05.mma.kind::mxf8f6f4.block_scale) against the oracle's scaled FP8
contraction, on ragged groups and every epilogue; non-power-of-two scales
are reported."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, require_gpu, to_np
from oracle.ffn import gemm_fp8, round_bf16, silu
from oracle.quant import dequant_1x128, quant_128x128, quant_1x128

# FP32 accumulation of the whole K reduction inside the tensor core: error
# bound relative to the sum of |products| (the FP32-scale kernel accumulates
# 128-element chunks there and promotes in registers: 1e-5)
MX_TOL = 1e-4

SIZES = [
    [0, 1, 127, 128, 129, 300, 0, 513],
    [256],
    [5, 0, 0, 0, 1000],
    [700, 300, 1000, 0, 257, 129, 513],
]


def _codes(rng, shape):
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] -= 1            # no NaN codes
    return c


def _pow2(rng, shape):
    return np.ldexp(1.0, rng.integers(-12, -4, shape)).astype(np.float32)


def _cuda(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


@gpu
@pytest.mark.parametrize("case", range(len(SIZES)))
@pytest.mark.parametrize("N,K", [(256, 128), (512, 384), (768, 1024), (256, 7168)])
@pytest.mark.parametrize("epi", ["bf16", "f32", "bf16_f32_last"])
def test_gemm_mx_epilogues(case, N, K, epi):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(case * 100 + N + K)
    sizes = SIZES[case]
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1]) + 70
    A, sa = _codes(rng, (rows, K)), _pow2(rng, (rows, K // 128))
    B, sb = _codes(rng, (G, N, K)), _pow2(rng, (G, N // 128, K // 128))
    o_d, A_d, sa_d, B_d, sb_d = _cuda(offsets, A, sa, B, sb)
    code = {"bf16": binding.MOE_EPI_BF16, "f32": binding.MOE_EPI_F32,
            "bf16_f32_last": binding.MOE_EPI_BF16_F32_LAST}[epi]
    dt = torch.float32 if epi == "f32" else torch.bfloat16
    out = torch.full((rows, N), -7.0, dtype=dt, device="cuda")
    last = torch.full((int(offsets[G] - offsets[G - 1]), N), -7.0, dtype=torch.float32, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, code, out, last if epi == "bf16_f32_last" else None,
                             block_scaled=True)
    binding.check_device_status()
    got = to_np(out).astype(np.float64)
    worst = 0.0
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        exact = gemm_fp8(A[r0:r1], sa[r0:r1], B[g], sb[g])
        mag = gemm_fp8(A[r0:r1] & 0x7F, sa[r0:r1], B[g] & 0x7F, sb[g])
        kind, rows_got = epi, got[r0:r1]
        if epi == "bf16_f32_last":
            if g == G - 1:
                kind, rows_got = "f32", to_np(last).astype(np.float64)
                assert np.all(got[r0:r1] == -7.0)
            else:
                kind = "bf16"
        err = np.abs(rows_got - exact)
        if kind == "bf16":
            assert np.all(err <= 2.0 ** -8 * np.abs(exact) + MX_TOL * mag + 1e-30), f"group {g}"
            assert np.mean(rows_got == round_bf16(exact)) > 0.99
        else:
            worst = max(worst, float((err / (mag + 1e-300)).max()))
            assert np.all(err <= MX_TOL * mag + 1e-30), f"group {g}: {(err / mag).max():.3e}"
    print(f"[mx-gemm] {epi} N={N} K={K} case={case}: worst |err| / sum|products| = {worst:.2e}")
    assert np.all(got[offsets[-1]:] == -7.0)


@gpu
@pytest.mark.parametrize("case", range(len(SIZES)))
@pytest.mark.parametrize("I,K", [(128, 256), (384, 7168)])
def test_gemm_mx_swiglu(case, I, K):
    """Gate/up GEMM + SwiGLU + power-of-two 1x128 requantisation of h."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(case + I + K)
    sizes = SIZES[case]
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1]) + 3
    xq, xs = quant_1x128(rng.standard_normal((rows, K)).astype(np.float32), "pow2")
    W1 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32), "pow2") for _ in range(G)]
    W3 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32), "pow2") for _ in range(G)]
    q1 = np.stack([w[0] for w in W1]); s1 = np.stack([w[1] for w in W1])
    q3 = np.stack([w[0] for w in W3]); s3 = np.stack([w[1] for w in W3])
    q1_d, s1_d, q3_d, s3_d, o_d, xq_d, xs_d = _cuda(q1, s1, q3, s3, offsets, xq, xs)
    q13, s13 = binding.pack_w13(q1_d, s1_d, q3_d, s3_d)
    hq = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
    hs = torch.full((rows, I // 128), -1.0, dtype=torch.float32, device="cuda")
    binding.grouped_gemm_fp8(o_d, xq_d, xs_d, q13, s13, binding.MOE_EPI_SWIGLU_FP8, hq, hs, block_scaled=True)
    binding.check_device_status()
    ghq, ghs = to_np(hq), to_np(hs)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        gate = gemm_fp8(xq[r0:r1], xs[r0:r1], q1[g], s1[g])
        up = gemm_fp8(xq[r0:r1], xs[r0:r1], q3[g], s3[g])
        h = (silu(gate) * up).astype(np.float32)
        rq, rs = quant_1x128(h, "pow2")
        assert np.all(np.frexp(ghs[r0:r1].astype(np.float64))[0] == 0.5), "h scales are powers of two"
        # the power-of-two scale changes only where h's amax sits within rounding of a boundary
        assert np.mean(ghs[r0:r1] == rs) > 0.99, f"scales of group {g}"
        assert np.mean(ghq[r0:r1] == rq) > 0.98
        dg = dequant_1x128(ghq[r0:r1], ghs[r0:r1])
        dr = dequant_1x128(rq, rs)
        # one E4M3 step of the larger of the two scales, plus the FP32 accumulation difference
        tol = 0.13 * np.abs(dr) + 2.0 ** -9 * np.repeat(np.maximum(rs, ghs[r0:r1]), 128, axis=1) * 1.01 + 1e-30
        assert np.all(np.abs(dg - dr) <= tol)
    assert np.all(ghq[offsets[-1]:] == 0x55) and np.all(ghs[offsets[-1]:] == -1.0)


@gpu
def test_gemm_mx_reports_non_power_of_two_scales():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(9)
    offsets = np.array([0, 200], np.int32)
    A, sa = _codes(rng, (200, 256)), _pow2(rng, (200, 2))
    B, sb = _codes(rng, (1, 256, 256)), _pow2(rng, (1, 2, 2))
    sa[17, 1] = np.float32(3.0 / 448)                  # not a power of two
    o_d, A_d, sa_d, B_d, sb_d = _cuda(offsets, A, sa, B, sb)
    out = torch.zeros((200, 256), dtype=torch.bfloat16, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, binding.MOE_EPI_BF16, out, block_scaled=True)
    with pytest.raises(binding.MoeError) as e:
        binding.check_device_status()
    assert e.value.code == 6
    binding.check_device_status()   # cleared
