"""GPU parity: FP8 quantisation kernels bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, require_gpu, to_np
from oracle.quant import quant_128x128, quant_1x128


def _activation(rows, cols, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device="cuda")
    x = x * torch.exp(torch.randn(rows, 1, generator=g, device="cuda") * 4)   # per-row magnitudes e^[-12, 12]
    x = x.to(torch.bfloat16)
    if rows >= 4 and cols >= 256:
        x[0, :128] = 0                                   # all-zero tile
        x[1, :128] = -0.0                                # negative zeros
        x[1, 5] = 3.0e-39                                # bf16 subnormal amax
        x[2, :128] = torch.tensor(1.0e38, dtype=torch.bfloat16)
        x[3, 128:256] = torch.tensor(-2.0 ** -133, dtype=torch.bfloat16)   # smallest subnormal
    return x


@gpu
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (256, 7168), (4096, 2048), (129, 1408)])
def test_quant_1x128_bit_exact(rows, cols):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    x = _activation(rows, cols, rows * 31 + cols)
    q, s = binding.quant_1x128(x)
    rq, rs = quant_1x128(to_np(x))
    assert np.array_equal(to_np(q), rq)
    assert np.array_equal(to_np(s).view(np.uint32), rs.view(np.uint32))


@gpu
def test_quant_1x128_full_width_prefill_input():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding, inputs
    from sparse_moe_layer_13_b300.configs import FULL
    x = inputs.gen_x(FULL, "cuda")
    q, s = binding.quant_1x128(x)
    rq, rs = quant_1x128(to_np(x))
    assert np.array_equal(to_np(q), rq)
    assert np.array_equal(to_np(s), rs)


@gpu
@pytest.mark.parametrize("batch,rows,cols", [(1, 128, 128), (3, 256, 384), (2, 2048, 1408)])
def test_quant_128x128_bit_exact(batch, rows, cols):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    g = torch.Generator(device="cuda")
    g.manual_seed(batch * 7 + rows)
    w = torch.randn(batch, rows, cols, generator=g, device="cuda") / 40
    w[0, :128, :128] = 0
    q, s = binding.quant_128x128(w)
    wn = to_np(w)
    for b in range(batch):
        rq, rs = quant_128x128(wn[b])
        assert np.array_equal(to_np(q[b]), rq)
        assert np.array_equal(to_np(s[b]), rs)


@gpu
def test_pack_w13_layout():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    I, d, b = 256, 256, 2
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    q1 = torch.randint(0, 126, (b, I, d), generator=g, device="cuda", dtype=torch.uint8)
    q3 = torch.randint(0, 126, (b, I, d), generator=g, device="cuda", dtype=torch.uint8)
    s1 = torch.rand(b, I // 128, d // 128, generator=g, device="cuda")
    s3 = torch.rand(b, I // 128, d // 128, generator=g, device="cuda")
    q13, s13 = binding.pack_w13(q1, s1, q3, s3)
    Q1, Q3, Q13 = to_np(q1), to_np(q3), to_np(q13)
    for j in range(I // 128):
        base = 256 * j
        assert np.array_equal(Q13[:, base:base + 64], Q1[:, 128 * j:128 * j + 64])
        assert np.array_equal(Q13[:, base + 64:base + 128], Q3[:, 128 * j:128 * j + 64])
        assert np.array_equal(Q13[:, base + 128:base + 192], Q1[:, 128 * j + 64:128 * j + 128])
        assert np.array_equal(Q13[:, base + 192:base + 256], Q3[:, 128 * j + 64:128 * j + 128])
        assert np.array_equal(to_np(s13)[:, 2 * j], to_np(s1)[:, j])
        assert np.array_equal(to_np(s13)[:, 2 * j + 1], to_np(s3)[:, j])
