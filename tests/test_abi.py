"""The C-ABI library loads without a GPU, exports every symbol its header
declares, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_moe_layer_13_b300 import binding
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_six_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_quant_fp8_1x128", "moe_grouped_gemm_fp8", "moe_combine",
              "moe_bias_update"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from sparse_moe_layer_13_b300 import binding
    for code, name in binding.STATUS.items():
        assert lib.moe_status_string(code).decode().startswith(name)
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"


def test_workspace_size_and_config_checks(lib):
    from sparse_moe_layer_13_b300 import binding
    from sparse_moe_layer_13_b300.configs import CONFIGS, MoEConfig
    for cfg in CONFIGS.values():
        assert binding.workspace_size(cfg) >= cfg.T * cfg.E * 4
    bad = [
        MoEConfig("b", T=8, d=200, E=16, I=128, K=2, G=4, M=2, gk=2, seed=0),    # d % 128
        MoEConfig("b", T=8, d=128, E=20, I=128, K=2, G=4, M=2, gk=2, seed=0),    # E % 16
        MoEConfig("b", T=8, d=128, E=16, I=128, K=2, G=4, M=5, gk=2, seed=0),    # M > G
        MoEConfig("b", T=8, d=128, E=16, I=128, K=9, G=4, M=2, gk=2, seed=0),    # K > M*E/G
        MoEConfig("b", T=8, d=128, E=16, I=128, K=2, G=4, M=2, gk=5, seed=0),    # gk > E/G
        MoEConfig("b", T=0, d=128, E=16, I=128, K=2, G=4, M=2, gk=2, seed=0),    # T < 1
    ]
    for cfg in bad:
        assert binding.workspace_size(cfg) == 0


def test_host_side_errors_return_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)          # aligned, never dereferenced: every call below fails its host checks
    odd = P(0x10001)
    assert lib.moe_quant_fp8_1x128(None, 4, 128, 128, fake, fake, None) == 1
    assert lib.moe_quant_fp8_1x128(fake, 4, 100, 128, fake, fake, None) == 2
    assert lib.moe_quant_fp8_1x128(odd, 4, 128, 128, fake, fake, None) == 1
    assert lib.moe_quant_fp8_128x128(fake, 1, 100, 128, fake, fake, None) == 2
    assert lib.moe_grouped_gemm_fp8(4, fake, 100, 200, 256, fake, fake, fake, fake, 0, fake, None, None) == 2
    assert lib.moe_grouped_gemm_fp8(4, fake, 100, 256, 200, fake, fake, fake, fake, 0, fake, None, None) == 2
    assert lib.moe_grouped_gemm_fp8(4, fake, 100, 256, 256, fake, fake, fake, fake, 7, fake, None, None) == 1
    assert lib.moe_grouped_gemm_fp8(4, fake, 100, 256, 256, fake, fake, fake, fake, 1, fake, None, None) == 1
    assert lib.moe_grouped_gemm_fp8(2000, fake, 100, 256, 256, fake, fake, fake, fake, 0, fake, None, None) == 2
    assert lib.moe_bias_update(0, 4, 2, fake, ctypes.c_float(0.1), fake, None) == 1
    assert lib.moe_combine(None, fake, fake, fake, fake, None, fake, None) == 1
    from sparse_moe_layer_13_b300 import binding
    from sparse_moe_layer_13_b300.configs import TINY
    c = binding.config_c(TINY)
    # workspace too small
    assert lib.moe_permute(ctypes.byref(c), fake, fake, fake, fake, None, fake, fake, fake, fake, fake, 16, None) == 3
    assert lib.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, fake, None, None, 0, None) == 3
    # router on weight planes: bad path enum, fused path beyond 256 experts, small workspace, null weight
    from sparse_moe_layer_13_b300.configs import MoEConfig
    big = binding.config_c(MoEConfig("e512", T=64, d=128, E=512, I=128, K=8, G=8, M=4, gk=2, seed=1))
    huge = 1 << 40
    assert lib.moe_route_planes(ctypes.byref(c), fake, fake, None, fake, fake, fake, None, 7, fake, huge, None) == 1
    assert lib.moe_route_planes(ctypes.byref(big), fake, fake, None, fake, fake, fake, None, 1, fake, huge, None) == 2
    assert lib.moe_route_planes(ctypes.byref(c), fake, fake, None, fake, fake, fake, None, 0, fake, 16, None) == 3
    assert lib.moe_route_planes(ctypes.byref(c), fake, None, None, fake, fake, fake, None, 0, fake, huge, None) == 1
    assert lib.moe_router_planes(None, 16, 256, fake, None) == 1


def test_backward_host_side_errors_return_before_launch(lib):
    """Every backward entry point rejects bad pointers, enums and shapes on the host."""
    from sparse_moe_layer_13_b300 import binding
    from sparse_moe_layer_13_b300.configs import TINY
    P = ctypes.c_void_p
    fake = P(0x10000)
    odd = P(0x10001)
    not32 = P(0x10010)         # 16-byte but not 32-byte aligned
    c = ctypes.byref(binding.config_c(TINY))
    # block transpose: null source, ldT < rows, rows not a multiple of 128
    assert lib.moe_transpose_fp8_blocks(None, fake, 1, 128, 128, fake, fake, 128, 128, None) == 1
    assert lib.moe_transpose_fp8_blocks(fake, fake, 1, 256, 128, fake, fake, 128, 128, None) == 1
    assert lib.moe_transpose_fp8_blocks(fake, fake, 1, 100, 128, fake, fake, 128, 128, None) == 2
    # combine / router backward: bad scale rule, config, workspace, alignment
    assert lib.moe_combine_backward(c, fake, fake, fake, fake, 5, fake, fake, fake, fake, None) == 1
    assert lib.moe_combine_backward(None, fake, fake, fake, fake, 0, fake, fake, fake, fake, None) == 1
    assert lib.moe_route_backward(c, None, fake, fake, fake, None, 0, None) == 3
    assert lib.moe_router_wgrad(c, odd, fake, fake, fake, fake, fake, None) == 1
    assert lib.moe_dx_combine(c, fake, fake, fake, fake, fake, None, fake, None) == 1
    # SwiGLU backward: ld_dh < I, I not a multiple of 128
    assert lib.moe_swiglu_backward(4, 256, fake, fake, 128, 0, fake, fake, None) == 1
    assert lib.moe_swiglu_backward(4, 100, fake, fake, 100, 0, fake, fake, None) == 2
    # 128x1 quantisers: columns, group count, ldq alignment, source strides
    assert lib.moe_quant_fp8_128x1_f32(fake, 128, 2, fake, 64, 100, 0, fake, 1024, fake, None) == 2
    assert lib.moe_quant_fp8_128x1_f32(fake, 128, 2000, fake, 64, 128, 0, fake, 1024, fake, None) == 2
    assert lib.moe_quant_fp8_128x1_f32(fake, 128, 2, fake, 64, 128, 0, fake, 1000, fake, None) == 1
    assert lib.moe_quant_fp8_128x1_f32(fake, 128, 2, fake, 64, 128, 3, fake, 1024, fake, None) == 1
    assert lib.moe_quant_fp8_128x1_fp8(fake, fake, 200, 2, fake, 64, 128, 0, fake, 1024, fake, None) == 1
    assert lib.moe_quant_fp8_128x1_bf16_rows(fake, 8, 128, None, None, 2, fake, 64, 128, 0, fake, 1024, fake,
                                            None) == 1
    # weight-gradient GEMM: M, N tiles, group count, output alignment
    assert lib.moe_grouped_wgrad_fp8(2, fake, 64, 512, 100, 256, fake, fake, fake, fake, fake, None) == 2
    assert lib.moe_grouped_wgrad_fp8(2, fake, 64, 512, 128, 128, fake, fake, fake, fake, fake, None) == 2
    assert lib.moe_grouped_wgrad_fp8(2000, fake, 64, 512, 128, 256, fake, fake, fake, fake, fake, None) == 2
    assert lib.moe_grouped_wgrad_fp8(2, fake, 64, 512, 128, 256, fake, fake, fake, fake, not32, None) == 1
    # the gate/up FP32 epilogue has no block-scaled variant
    assert lib.moe_grouped_gemm_fp8_mx(4, fake, 100, 256, 256, fake, fake, fake, fake, 4, fake, None, None) == 2


def test_expert_parallel_host_side_checks(lib):
    """Expert-parallel entry points: packed row size, workspace query, and rejects of a
    rank count that does not split the experts, bad ranks, null pointers and small
    workspaces, all before any launch."""
    from sparse_moe_layer_13_b300 import binding
    from sparse_moe_layer_13_b300.configs import TINY
    P = ctypes.c_void_p
    fake = P(0x10000)
    c = ctypes.byref(binding.config_c(TINY))            # E = 16, K = 4, d = 256
    # 256 code bytes + 2 scales * 4 + 4 ids * 4 + 4 gates * 4 = 296 -> 304
    assert lib.moe_ep_row_bytes(256, 4) == 304
    assert lib.moe_ep_row_bytes(7168, 8) == 7168 + 224 + 64
    assert lib.moe_ep_row_bytes(100, 4) == 0 and lib.moe_ep_row_bytes(256, 17) == 0
    assert lib.moe_ep_workspace_size(c, 3, 256) == 0      # 16 experts do not split over 3 ranks
    assert lib.moe_ep_workspace_size(c, 4, 256) > 0
    big = 1 << 40
    assert lib.moe_ep_dispatch(c, 3, fake, fake, fake, fake, None, fake, fake, fake, fake, fake, big, None) == 2
    assert lib.moe_ep_dispatch(c, 4, None, fake, fake, fake, None, fake, fake, fake, fake, fake, big, None) == 1
    assert lib.moe_ep_dispatch(c, 4, fake, fake, fake, fake, None, fake, fake, fake, fake, fake, 16, None) == 3
    assert lib.moe_ep_receive(c, 4, 4, 10, fake, fake, None, fake, fake, fake, fake, fake, big, None) == 2
    assert lib.moe_ep_receive(c, 4, 0, 10, None, fake, None, fake, fake, fake, fake, fake, big, None) == 1
    assert lib.moe_ep_receive(c, 4, 0, 10, fake, fake, None, fake, fake, fake, fake, fake, 16, None) == 3
    assert lib.moe_ep_partial(c, 5, None, fake, fake, 10, fake, None) == 1
    assert lib.moe_ep_combine(c, None, fake, 10, fake, None, fake, None) == 1
    assert lib.moe_ep_combine(c, fake, None, 10, fake, None, fake, None) == 1
