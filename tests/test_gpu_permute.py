"""GPU parity: histogram, offsets and stable permutation bit-exact against the
oracle's counting sort; gathered rows bit-exact; corrupt indices reported."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, require_gpu, to_np
from oracle.permute import histogram, permute as oracle_permute
from oracle.quant import quant_1x128
from sparse_moe_layer_13_b300.configs import CONFIGS, MoEConfig


def _check(cfg, idx_np, seed=0, gather_rows=True):
    from sparse_moe_layer_13_b300 import binding, inputs
    x = inputs.gen_x(cfg, "cuda", step=seed)
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    xq, xs = binding.quant_1x128(x)
    out = binding.permute(cfg, idx, xq, xs, want_counts=True, gather_rows=gather_rows)
    binding.check_device_status()
    offsets, sorted_token, row_of = oracle_permute(idx_np, cfg.E)
    T, K = cfg.T, cfg.K
    got_off = to_np(out["offsets"])
    assert np.array_equal(got_off[:cfg.E + 1], offsets)
    assert got_off[cfg.E + 1] == T * K + T
    assert np.array_equal(to_np(out["counts"]), histogram(idx_np, cfg.E))
    src = np.concatenate([sorted_token, np.arange(T)])      # the shared expert's rows read token t
    assert np.array_equal(to_np(out["sorted_token"]), src)
    assert np.array_equal(to_np(out["row_of"]), row_of)
    if not gather_rows:
        assert out["xq_perm"] is None
        return
    rq, rs = quant_1x128(to_np(x))
    assert np.array_equal(to_np(out["xq_perm"]), rq[src])
    assert np.array_equal(to_np(out["xs_perm"]), rs[src])


def _random_idx(T, E, K, seed, p=None):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)])


@gpu
@pytest.mark.parametrize("name", ["tiny", "mid", "full", "decode"])
def test_permute_workloads(name):
    require_gpu()
    cfg = CONFIGS[name]
    _check(cfg, _random_idx(cfg.T, cfg.E, cfg.K, 1))


@gpu
@pytest.mark.parametrize("name", ["tiny", "full"])
def test_permute_without_row_gather(name):
    require_gpu()
    cfg = CONFIGS[name]
    _check(cfg, _random_idx(cfg.T, cfg.E, cfg.K, 7), gather_rows=False)


@gpu
def test_permute_hot_expert_and_empty_experts():
    require_gpu()
    cfg = MoEConfig("hot", T=1000, d=256, E=64, I=128, K=4, G=8, M=4, gk=1, seed=3)
    rng = np.random.default_rng(2)
    others = np.array([0, 1, 2, 3, 4, 6, 7])
    idx = np.stack([np.concatenate([[5], rng.choice(others, 3, replace=False)]) for _ in range(cfg.T)])
    _check(cfg, idx)                            # expert 5 in every token, experts 8..63 empty


@gpu
@pytest.mark.parametrize("T,E,K,G,M", [(1, 16, 1, 4, 2), (257, 16, 4, 4, 2), (513, 1024, 16, 32, 4),
                                       (3000, 256, 8, 8, 4)])
def test_permute_ragged_and_extremes(T, E, K, G, M):
    require_gpu()
    cfg = MoEConfig("r", T=T, d=256, E=E, I=128, K=K, G=G, M=M, gk=1, seed=4)
    zipf = 1.0 / np.arange(1, E + 1) ** 1.1
    _check(cfg, _random_idx(T, E, K, 5, p=zipf / zipf.sum()))


@gpu
def test_permute_reports_out_of_range_expert():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    cfg = CONFIGS["tiny"]
    idx = _random_idx(cfg.T, cfg.E, cfg.K, 6)
    idx[10, 2] = cfg.E            # corrupt
    x = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    xq, xs = binding.quant_1x128(x)
    binding.permute(cfg, torch.from_numpy(idx.astype(np.int32)).cuda(), xq, xs)
    with pytest.raises(binding.MoeError) as e:
        binding.check_device_status()
    assert e.value.code == 6
    binding.check_device_status()   # cleared
