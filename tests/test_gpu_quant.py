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
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (256, 7168), (4096, 2048), (129, 1408)])
def test_quant_1x128_bit_exact(rows, cols, rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    x = _activation(rows, cols, rows * 31 + cols)
    q, s = binding.quant_1x128(x, rule=rule)
    rq, rs = quant_1x128(to_np(x), rule)
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
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
@pytest.mark.parametrize("batch,rows,cols", [(1, 128, 128), (3, 256, 384), (2, 2048, 1408)])
def test_quant_128x128_bit_exact(batch, rows, cols, rule):
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    g = torch.Generator(device="cuda")
    g.manual_seed(batch * 7 + rows)
    w = torch.randn(batch, rows, cols, generator=g, device="cuda") / 40
    w[0, :128, :128] = 0
    q, s = binding.quant_128x128(w, rule=rule)
    wn = to_np(w)
    for b in range(batch):
        rq, rs = quant_128x128(wn[b], rule)
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


def _scatter_case(T, d, E, K, seed):
    from sparse_moe_layer_13_b300.configs import MoEConfig
    cfg = MoEConfig("scatter", T=T, d=d, E=E, I=128, K=K, G=E // 16 if E >= 16 else 1, M=1, gk=1, seed=seed)
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    return cfg, idx


@gpu
@pytest.mark.parametrize("rule", ["fp32", "pow2"])
@pytest.mark.parametrize("T,d,E,K", [(1, 128, 16, 1), (37, 256, 16, 4), (300, 7168, 256, 8), (1000, 1408, 64, 16)])
def test_quant_1x128_scatter_bit_exact(T, d, E, K, rule):
    """Codes and scales land in grouped order: row row_of[t][k] and the
    shared-expert row T*K + t each hold token t's quantised row."""
    require_gpu()
    from oracle.permute import permute as oracle_permute
    from sparse_moe_layer_13_b300 import binding
    cfg, idx = _scatter_case(T, d, E, K, T + d)
    _, sorted_token, row_of = oracle_permute(idx, E)
    x = _activation(T, d, T * 7 + d)
    q, s = binding.quant_1x128_scatter(cfg, x, torch.from_numpy(row_of.astype(np.int32)).cuda(), rule=rule)
    binding.check_device_status()
    rq, rs = quant_1x128(to_np(x), rule)
    src = np.concatenate([sorted_token, np.arange(T)])
    assert np.array_equal(to_np(q), rq[src])
    assert np.array_equal(to_np(s).view(np.uint32), rs[src].view(np.uint32))


@gpu
def test_quant_1x128_scatter_reports_bad_row():
    require_gpu()
    from oracle.permute import permute as oracle_permute
    from sparse_moe_layer_13_b300 import binding
    cfg, idx = _scatter_case(64, 256, 16, 4, 9)
    _, sorted_token, row_of = oracle_permute(idx, 16)
    row_of = row_of.astype(np.int32)
    bad = row_of[5, 2]
    row_of[5, 2] = cfg.T * cfg.K               # the first shared-expert row: not a routed row
    x = _activation(cfg.T, cfg.d, 3)
    q = torch.full((cfg.rows, cfg.d), 0x55, dtype=torch.uint8, device="cuda")
    s = torch.full((cfg.rows, cfg.d // 128), -1.0, dtype=torch.float32, device="cuda")
    binding.quant_1x128_scatter(cfg, x, torch.from_numpy(row_of).cuda(), q, s)
    with pytest.raises(binding.MoeError) as e:
        binding.check_device_status()
    assert e.value.code == 6
    binding.check_device_status()   # cleared
    assert torch.all(q[bad] == 0x55)           # the slot the bad entry should have filled stays untouched
    rq, _ = quant_1x128(to_np(x))
    assert np.array_equal(to_np(q[cfg.T * cfg.K]), rq[0])   # shared row of token 0 written normally
