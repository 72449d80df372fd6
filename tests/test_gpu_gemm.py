"""GPU parity: grouped FP8 GEMM (tcgen05) against the oracle's scaled FP8
contraction, on ragged groups (empty, single-row, tile-straddling), every
epilogue, row-gathered A, and corrupt offsets or row indices."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, require_gpu, to_np
from oracle import e4m3
from oracle.ffn import gemm_fp8, round_bf16, silu
from oracle.quant import dequant_1x128, quant_1x128


def _codes(rng, shape):
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] -= 1            # no NaN codes
    return c


def _problem(sizes, N, K, seed, trailing=0):
    rng = np.random.default_rng(seed)
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1]) + trailing
    A = _codes(rng, (rows, K))
    sa = rng.uniform(0.5, 2.0, (rows, K // 128)).astype(np.float32) / 448
    B = _codes(rng, (G, N, K))
    sb = rng.uniform(0.5, 2.0, (G, N // 128, K // 128)).astype(np.float32) / 448
    return offsets, A, sa, B, sb


def _cuda(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


SIZES = [
    [0, 1, 127, 128, 129, 300, 0, 513],
    [256],
    [5, 0, 0, 0, 1000],
    # larger groups: several row tiles each, ragged last tiles, an empty
    # group and groups of one tile plus one row
    [700, 300, 1000, 0, 257, 129, 513],
]


@gpu
@pytest.mark.parametrize("case", range(len(SIZES)))
@pytest.mark.parametrize("N,K", [(256, 128), (512, 384), (768, 1024)])
@pytest.mark.parametrize("epi", ["bf16", "f32", "bf16_f32_last"])
def test_gemm_plain_epilogues(case, N, K, epi):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    offsets, A, sa, B, sb = _problem(SIZES[case], N, K, seed=case * 100 + N + K, trailing=70)
    o_d, A_d, sa_d, B_d, sb_d = _cuda(offsets, A, sa, B, sb)
    code = {"bf16": binding.MOE_EPI_BF16, "f32": binding.MOE_EPI_F32,
            "bf16_f32_last": binding.MOE_EPI_BF16_F32_LAST}[epi]
    dt = torch.float32 if epi == "f32" else torch.bfloat16
    out = torch.full((A.shape[0], N), -7.0, dtype=dt, device="cuda")
    G = len(offsets) - 1
    last = torch.full((int(offsets[G] - offsets[G - 1]), N), -7.0, dtype=torch.float32, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, code, out, last if epi == "bf16_f32_last" else None)
    binding.check_device_status()
    got = to_np(out).astype(np.float64)
    absA, absB = A & 0x7F, B & 0x7F
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        exact = gemm_fp8(A[r0:r1], sa[r0:r1], B[g], sb[g])
        mag = gemm_fp8(absA[r0:r1], sa[r0:r1], absB[g], sb[g])   # sum of |products|: the FP32 error scale
        kind = epi
        rows_got = got[r0:r1]
        if epi == "bf16_f32_last":
            if g == G - 1:
                kind = "f32"
                rows_got = to_np(last).astype(np.float64)
                assert np.all(got[r0:r1] == -7.0)          # the last group goes only to the FP32 output
            else:
                kind = "bf16"
        err = np.abs(rows_got - exact)
        if kind == "bf16":
            assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 1e-5 * mag + 1e-30), f"group {g}"
            assert np.mean(rows_got == round_bf16(exact)) > 0.99
        else:
            assert np.all(err <= 1e-5 * mag + 1e-30), f"group {g}: {(err / mag).max():.3e}"
    assert np.all(got[offsets[-1]:] == -7.0)       # rows outside every group untouched


@gpu
@pytest.mark.parametrize("case", range(len(SIZES)))
@pytest.mark.parametrize("I,K", [(128, 256), (384, 512)])
def test_gemm_swiglu_epilogue(case, I, K):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(case + I)
    sizes = SIZES[case]
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1]) + 3
    # realistic magnitudes: quantise N(0,1) activations and N(0,1/K) weights with the oracle
    xq, xs = quant_1x128(rng.standard_normal((rows, K)).astype(np.float32))
    from oracle.quant import quant_128x128
    W1 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32)) for _ in range(G)]
    W3 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32)) for _ in range(G)]
    q1 = np.stack([w[0] for w in W1]); s1 = np.stack([w[1] for w in W1])
    q3 = np.stack([w[0] for w in W3]); s3 = np.stack([w[1] for w in W3])
    q1_d, s1_d, q3_d, s3_d, o_d, xq_d, xs_d = _cuda(q1, s1, q3, s3, offsets, xq, xs)
    q13, s13 = binding.pack_w13(q1_d, s1_d, q3_d, s3_d)
    hq = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
    hs = torch.full((rows, I // 128), -1.0, dtype=torch.float32, device="cuda")
    binding.grouped_gemm_fp8(o_d, xq_d, xs_d, q13, s13, binding.MOE_EPI_SWIGLU_FP8, hq, hs)
    binding.check_device_status()
    ghq, ghs = to_np(hq), to_np(hs)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        gate = gemm_fp8(xq[r0:r1], xs[r0:r1], q1[g], s1[g])
        up = gemm_fp8(xq[r0:r1], xs[r0:r1], q3[g], s3[g])
        h = (silu(gate) * up).astype(np.float32)
        rq, rs = quant_1x128(h)
        assert np.allclose(ghs[r0:r1], rs, rtol=1e-5, atol=0), f"scales of group {g}"
        assert np.mean(ghq[r0:r1] == rq) > 0.99
        dg = dequant_1x128(ghq[r0:r1], ghs[r0:r1])
        dr = dequant_1x128(rq, rs)
        tol = 0.13 * np.abs(dr) + 2.0 ** -9 * np.repeat(rs, 128, axis=1) * 1.01 + 1e-30
        assert np.all(np.abs(dg - dr) <= tol)
    assert np.all(ghq[offsets[-1]:] == 0x55) and np.all(ghs[offsets[-1]:] == -1.0)


def _row_index(rng, rows, a_rows):
    """Grouped row -> A row: a permutation of the A rows, then repeats, as a
    token-to-expert gather makes (every token read K + 1 times)."""
    idx = np.concatenate([rng.permutation(a_rows), rng.integers(0, a_rows, max(0, rows - a_rows))])[:rows]
    return idx.astype(np.int32)


@gpu
@pytest.mark.parametrize("case", range(len(SIZES)))
@pytest.mark.parametrize("N,K,a_rows", [(256, 128, 7), (512, 384, 1000), (768, 1024, 333)])
@pytest.mark.parametrize("epi", ["bf16", "f32"])
def test_gemm_gathered_rows(case, N, K, a_rows, epi):
    """A rows fetched by index give exactly the GEMM of the gathered matrix."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(case * 7 + K)
    sizes = SIZES[case]
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    A = _codes(rng, (a_rows, K))
    sa = rng.uniform(0.5, 2.0, (a_rows, K // 128)).astype(np.float32) / 448
    B = _codes(rng, (G, N, K))
    sb = rng.uniform(0.5, 2.0, (G, N // 128, K // 128)).astype(np.float32) / 448
    ridx = _row_index(rng, rows, a_rows)
    o_d, A_d, sa_d, B_d, sb_d, ri_d = _cuda(offsets, A, sa, B, sb, ridx)
    code = binding.MOE_EPI_F32 if epi == "f32" else binding.MOE_EPI_BF16
    dt = torch.float32 if epi == "f32" else torch.bfloat16
    out = torch.full((rows + 5, N), -7.0, dtype=dt, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, code, out, row_index=ri_d)
    binding.check_device_status()
    got = to_np(out).astype(np.float64)
    Ag, sag = A[ridx], sa[ridx]
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        exact = gemm_fp8(Ag[r0:r1], sag[r0:r1], B[g], sb[g])
        mag = gemm_fp8(Ag[r0:r1] & 0x7F, sag[r0:r1], B[g] & 0x7F, sb[g])
        err = np.abs(got[r0:r1] - exact)
        if epi == "bf16":
            assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 1e-5 * mag + 1e-30), f"group {g}"
            assert np.mean(got[r0:r1] == round_bf16(exact)) > 0.99
        else:
            assert np.all(err <= 1e-5 * mag + 1e-30), f"group {g}: {(err / mag).max():.3e}"
    assert np.all(got[rows:] == -7.0)


@gpu
def test_gemm_gathered_swiglu_matches_plain():
    """Gathered A rows through the SwiGLU epilogue give bit-identical h to the
    same GEMM on the pre-gathered matrix (same tile order, same arithmetic)."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    from oracle.quant import quant_128x128
    rng = np.random.default_rng(11)
    I, K, G, a_rows = 384, 512, 4, 500
    sizes = [300, 0, 129, 1100]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    xq, xs = quant_1x128(rng.standard_normal((a_rows, K)).astype(np.float32))
    W1 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32)) for _ in range(G)]
    W3 = [quant_128x128((rng.standard_normal((I, K)) / np.sqrt(K)).astype(np.float32)) for _ in range(G)]
    q1 = np.stack([w[0] for w in W1]); s1 = np.stack([w[1] for w in W1])
    q3 = np.stack([w[0] for w in W3]); s3 = np.stack([w[1] for w in W3])
    ridx = _row_index(rng, rows, a_rows)
    q1_d, s1_d, q3_d, s3_d, o_d, xq_d, xs_d, ri_d, xqg_d, xsg_d = _cuda(q1, s1, q3, s3, offsets, xq, xs, ridx,
                                                                       xq[ridx], xs[ridx])
    q13, s13 = binding.pack_w13(q1_d, s1_d, q3_d, s3_d)
    outs = []
    for gathered in (False, True):
        hq = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
        hs = torch.full((rows, I // 128), -1.0, dtype=torch.float32, device="cuda")
        if gathered:
            binding.grouped_gemm_fp8(o_d, xq_d, xs_d, q13, s13, binding.MOE_EPI_SWIGLU_FP8, hq, hs, row_index=ri_d)
        else:
            binding.grouped_gemm_fp8(o_d, xqg_d, xsg_d, q13, s13, binding.MOE_EPI_SWIGLU_FP8, hq, hs)
        binding.check_device_status()
        outs.append((to_np(hq), to_np(hs)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


@gpu
def test_gemm_reports_out_of_range_row_index():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    offsets, A, sa, B, sb = _problem([10, 20, 30], 256, 128, seed=2)
    ridx = np.arange(60, dtype=np.int32)
    ridx[17] = A.shape[0]           # one past the last A row
    o_d, A_d, sa_d, B_d, sb_d, ri_d = _cuda(offsets, A, sa, B, sb, ridx)
    out = torch.zeros((60, 256), dtype=torch.bfloat16, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, binding.MOE_EPI_BF16, out, row_index=ri_d)
    with pytest.raises(binding.MoeError) as e:
        binding.check_device_status()
    assert e.value.code == 6
    binding.check_device_status()   # cleared


@gpu
def test_gemm_reports_corrupt_offsets():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    offsets, A, sa, B, sb = _problem([10, 20, 30], 256, 128, seed=1)
    bad = offsets.copy()
    bad[2] = 5                      # not monotone
    o_d, A_d, sa_d, B_d, sb_d = _cuda(bad, A, sa, B, sb)
    out = torch.full((A.shape[0], 256), 3.0, dtype=torch.bfloat16, device="cuda")
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, binding.MOE_EPI_BF16, out)
    with pytest.raises(binding.MoeError) as e:
        binding.check_device_status()
    assert e.value.code == 6
    assert torch.all(out == 3.0)    # nothing written
    bad = offsets.copy()
    bad[-1] = A.shape[0] + 1        # past the last row
    o_d = _cuda(bad)[0]
    binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, binding.MOE_EPI_BF16, out)
    with pytest.raises(binding.MoeError):
        binding.check_device_status()


@gpu
@pytest.mark.parametrize("K", [2048, 7168])
def test_gemm_f32_within_evaluation_bound(K):
    """Pins the evaluation bound the oracle's gradient and output budgets rest on
    (oracle/bounds.py, gemm_bound): every FP32 output of the grouped GEMM lies within the
    bound of the exact chunk-promoted sum, on operands quantised from Gaussian values as the
    layer's are (1x128 activations, 128x128 weight blocks)."""
    require_gpu()
    from oracle.quant import quant_128x128
    from sparse_moe_layer_13_b300 import binding
    rng = np.random.default_rng(K)
    sizes = [300, 0, 129, 512]
    N = 512
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    A, sa = quant_1x128(rng.standard_normal((rows, K)).astype(np.float32))
    Bq, sb = zip(*(quant_128x128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
                   for _ in sizes))
    B, sb = np.stack(Bq), np.stack(sb)
    o_d, A_d, sa_d, B_d, sb_d = _cuda(offsets, A, sa, B, sb)
    out, _ = binding.grouped_gemm_fp8(o_d, A_d, sa_d, B_d, sb_d, binding.MOE_EPI_F32)
    binding.check_device_status()
    got = to_np(out).astype(np.float64)
    worst = 0.0
    for g in range(len(sizes)):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        exact, bound = gemm_fp8(A[r0:r1], sa[r0:r1], B[g], sb[g], with_bound=True)
        ratio = np.abs(got[r0:r1] - exact) / bound
        worst = max(worst, float(ratio.max()))
        assert (ratio <= 1.0).all(), f"group {g}: {int((ratio > 1).sum())} outputs beyond the bound"
    print(f"[bound] K={K}: worst |error| / gemm_bound = {worst:.3f}")


def _off16(t):
    """The same values in a buffer whose first element sits 4 bytes past a 16-byte boundary."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = flat[1:].view(t.shape)
    v.copy_(t)
    return v


@gpu
@pytest.mark.parametrize("K", [512, 1024, 7168, 8704])
@pytest.mark.parametrize("epi", ["bf16", "swiglu", "bf16_f32_last", "f32", "gateup_f32"])
@pytest.mark.parametrize("gather", [False, True])
def test_gemm_scale_paths_agree(K, epi, gather):
    """The chunk scales reach the promotion either from registers plus a weight-scale row
    staged once per tile (16-byte aligned scale arrays, K/128 a multiple of 4 and at most 64)
    or through the per-chunk shared-memory ring (every other case). Both take the same FP32
    products in the same order, so the outputs agree bit for bit; scale arrays 4 bytes off a
    16-byte boundary force the ring. K = 8704 (68 chunks) takes the ring either way."""
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    sizes = [700, 300, 1000, 0, 257, 129, 513]
    N = 512
    offsets, A, sa, B, sb = _problem(sizes, N, K, seed=K + len(epi) + gather, trailing=5)
    rng = np.random.default_rng(K)
    rows = int(offsets[-1])
    ridx = _row_index(rng, rows, A.shape[0]) if gather else None
    o_d, A_d, sa_d, B_d, sb_d = _cuda(offsets, A, sa, B, sb)
    ri_d = _cuda(ridx)[0] if gather else None
    G = len(sizes)
    last_rows = int(offsets[G] - offsets[G - 1])
    outs = []
    for sa_x, sb_x in ((sa_d, sb_d), (_off16(sa_d), _off16(sb_d))):
        if epi == "swiglu":
            out = torch.full((rows, N // 2), 0x55, dtype=torch.uint8, device="cuda")
            aux = torch.full((rows, N // 256), -1.0, dtype=torch.float32, device="cuda")
            code = binding.MOE_EPI_SWIGLU_FP8
        elif epi in ("f32", "gateup_f32"):
            out = torch.full((rows, N), -7.0, dtype=torch.float32, device="cuda")
            aux = None
            code = binding.MOE_EPI_F32 if epi == "f32" else binding.MOE_EPI_GATEUP_F32
        else:
            out = torch.full((rows, N), -7.0, dtype=torch.bfloat16, device="cuda")
            aux = torch.full((last_rows, N), -7.0, dtype=torch.float32, device="cuda") if epi != "bf16" else None
            code = binding.MOE_EPI_BF16 if epi == "bf16" else binding.MOE_EPI_BF16_F32_LAST
        binding.grouped_gemm_fp8(o_d, A_d, sa_x, B_d, sb_x, code, out, aux, last_rows=last_rows, row_index=ri_d)
        binding.check_device_status()
        outs.append([to_np(out.view(torch.uint8) if out.dtype == torch.bfloat16 else out)] +
                    ([to_np(aux)] if aux is not None else []))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
