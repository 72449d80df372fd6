"""ctypes binding of libmoe_b300.so (C ABI declared in include/moe_b300.h).

Argument marshalling only: every wrapper checks dtypes, devices and
contiguity, allocates outputs with torch when the caller gives none, and
passes raw pointers plus the current CUDA stream to the library. There is
no fallback: if the shared library is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_NAME = "libmoe_b300.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

MOE_EPI_BF16 = 0
MOE_EPI_SWIGLU_FP8 = 1
MOE_EPI_F32 = 2
MOE_EPI_BF16_F32_LAST = 3
MOE_EPI_GATEUP_F32 = 4

STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_CHECK", 7: "MOE_ERR_NO_DEVICE",
}

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIG = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_check_device_status": (ctypes.c_int, [_P]),
    "moe_workspace_size": (ctypes.c_size_t, [_P]),
    "moe_route": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_router_planes": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "moe_route_planes": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, ctypes.c_size_t, _P]),
    "moe_quant_fp8_1x128": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "moe_quant_fp8_128x128": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "moe_pack_w13": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "moe_permute": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_permute_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_gemm_fp8": (ctypes.c_int, [_I32, _P, _I64, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P, _P]),
    "moe_grouped_gemm_fp8_gather": (ctypes.c_int, [_I32, _P, _I64, _I32, _I32, _P, _P, _I64, _P, _P, _P, _I32, _P, _P,
                                                   _P]),
    "moe_quant_fp8_1x128_scatter": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "moe_quant_fp8_1x128_rule": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _P]),
    "moe_quant_fp8_1x128_scatter_rule": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _P]),
    "moe_quant_fp8_128x128_rule": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _P]),
    "moe_grouped_gemm_fp8_mx": (ctypes.c_int, [_I32, _P, _I64, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P, _P]),
    "moe_balance_loss": (ctypes.c_int, [_P, _P, _P, _I32, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_bias_update": (ctypes.c_int, [_I32, _I32, _I32, _P, ctypes.c_float, _P, _P]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _P]),
    "moe_transpose_fp8_blocks": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P, _I64, _I64, _P]),
    "moe_combine_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P]),
    "moe_route_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_router_wgrad": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_swiglu_backward": (ctypes.c_int, [_I64, _I32, _P, _P, _I64, _I32, _P, _P, _P]),
    "moe_dx_combine": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_quant_fp8_128x1_f32": (ctypes.c_int, [_P, _I64, _I32, _P, _I64, _I32, _I32, _P, _I64, _P, _P]),
    "moe_quant_fp8_128x1_fp8": (ctypes.c_int, [_P, _P, _I64, _I32, _P, _I64, _I32, _I32, _P, _I64, _P, _P]),
    "moe_quant_fp8_128x1_bf16_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I32, _P, _I64, _I32, _I32, _P, _I64, _P,
                                                     _P]),
    "moe_grouped_wgrad_fp8": (ctypes.c_int, [_I32, _P, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "moe_ep_row_bytes": (ctypes.c_int64, [_I32, _I32]),
    "moe_ep_workspace_size": (ctypes.c_size_t, [_P, _I32, _I64]),
    "moe_ep_dispatch": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_ep_receive": (ctypes.c_int, [_P, _I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_ep_partial": (ctypes.c_int, [_P, _I64, _P, _P, _P, _I64, _P, _P]),
    "moe_ep_combine": (ctypes.c_int, [_P, _P, _P, _I64, _P, _P, _P, _P]),
}


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class MoEConfigC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "E", "I", "K", "G", "M", "gk")]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raise if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{LIB_NAME} is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIG.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _call(name: str, *args) -> None:
    rc = getattr(load(), name)(*args)
    if rc != 0:
        raise MoeError(name, rc)


SCALE_RULES = {"fp32": 0, "pow2": 1}     # moe_scale_rule


def _rule(rule: str) -> int:
    if rule not in SCALE_RULES:
        raise ValueError(f"scale rule: {rule!r}")
    return SCALE_RULES[rule]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, shape=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def config_c(cfg) -> MoEConfigC:
    return MoEConfigC(*cfg.abi())


def version() -> str:
    return load().moe_version().decode()


def check_device_status() -> None:
    rc = load().moe_check_device_status(_stream())
    if rc != 0:
        raise MoeError("device status", rc)


def selftest_wait_timeout(limit_us: int) -> int:
    return load().moe_selftest_wait_timeout(limit_us, _stream())


def workspace_size(cfg) -> int:
    c = config_c(cfg)
    return load().moe_workspace_size(ctypes.byref(c))


def route(cfg, x, Wr, bias, logit_offset=None, workspace=None, idx=None, gate=None, counts=None, want_counts=False):
    dev = x.device
    _need(x, torch.bfloat16, "x", (cfg.T, cfg.d))
    _need(Wr, torch.float32, "Wr", (cfg.E, cfg.d))
    _need(bias, torch.float32, "bias", (cfg.E,))
    if logit_offset is not None:
        _need(logit_offset, torch.float32, "logit_offset", (cfg.E,))
    idx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev) if idx is None else idx
    gate = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device=dev) if gate is None else gate
    if want_counts and counts is None:
        counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=dev)
    c = config_c(cfg)
    _call("moe_route", ctypes.byref(c), _ptr(x), _ptr(Wr), _ptr(logit_offset), _ptr(bias), _ptr(idx), _ptr(gate),
          _ptr(counts), _ptr(workspace), workspace.numel(), _stream())
    return idx, gate, counts


ROUTE_PATHS = {"auto": 0, "fused": 1, "split": 2}


def router_planes(Wr, planes=None):
    """Wr f32 [E][d] -> the three bf16 planes [3][E][d] (moe_router_planes)."""
    _need(Wr, torch.float32, "Wr")
    E, d = Wr.shape
    planes = torch.empty(3, E, d, dtype=torch.bfloat16, device=Wr.device) if planes is None else planes
    _need(planes, torch.bfloat16, "planes", (3, E, d))
    _call("moe_router_planes", _ptr(Wr), E, d, _ptr(planes), _stream())
    return planes


def route_planes(cfg, x, planes, bias, logit_offset=None, workspace=None, idx=None, gate=None, counts=None,
                 want_counts=False, path="auto"):
    """moe_route_planes: the router on pre-split weight planes, on the kernel path `path`
    ("auto", "fused" or "split")."""
    dev = x.device
    _need(x, torch.bfloat16, "x", (cfg.T, cfg.d))
    _need(planes, torch.bfloat16, "planes", (3, cfg.E, cfg.d))
    _need(bias, torch.float32, "bias", (cfg.E,))
    if logit_offset is not None:
        _need(logit_offset, torch.float32, "logit_offset", (cfg.E,))
    idx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev) if idx is None else idx
    gate = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device=dev) if gate is None else gate
    if want_counts and counts is None:
        counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=dev)
    c = config_c(cfg)
    _call("moe_route_planes", ctypes.byref(c), _ptr(x), _ptr(planes), _ptr(logit_offset), _ptr(bias), _ptr(idx),
          _ptr(gate), _ptr(counts), ROUTE_PATHS[path], _ptr(workspace), workspace.numel(), _stream())
    return idx, gate, counts


def quant_1x128(x, q=None, scale=None, rule="fp32"):
    _need(x, torch.bfloat16, "x")
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device) if q is None else q
    scale = torch.empty(rows, cols // 128, dtype=torch.float32, device=x.device) if scale is None else scale
    _call("moe_quant_fp8_1x128_rule", _ptr(x), rows, cols, cols, _rule(rule), _ptr(q), _ptr(scale), _stream())
    return q, scale


def quant_1x128_scatter(cfg, x, row_of, xq_perm=None, xs_perm=None, rule="fp32"):
    """Quantise tokens x [T][d] straight into grouped rows: row_of[t][k] and T*K + t."""
    _need(x, torch.bfloat16, "x", (cfg.T, cfg.d))
    _need(row_of, torch.int32, "row_of", (cfg.T, cfg.K))
    rows = cfg.rows
    xq_perm = torch.empty(rows, cfg.d, dtype=torch.uint8, device=x.device) if xq_perm is None else xq_perm
    xs_perm = torch.empty(rows, cfg.d // 128, dtype=torch.float32, device=x.device) if xs_perm is None else xs_perm
    _need(xq_perm, torch.uint8, "xq_perm", (rows, cfg.d))
    _need(xs_perm, torch.float32, "xs_perm", (rows, cfg.d // 128))
    c = config_c(cfg)
    _call("moe_quant_fp8_1x128_scatter_rule", ctypes.byref(c), _ptr(x), _ptr(row_of), _rule(rule), _ptr(xq_perm),
          _ptr(xs_perm), _stream())
    return xq_perm, xs_perm


def quant_128x128(w, q=None, scale=None, rule="fp32"):
    """w float32 [rows][cols] or [batch][rows][cols]."""
    _need(w, torch.float32, "w")
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    b, rows, cols = w3.shape
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device) if q is None else q
    sshape = (rows // 128, cols // 128) if w.dim() == 2 else (b, rows // 128, cols // 128)
    scale = torch.empty(sshape, dtype=torch.float32, device=w.device) if scale is None else scale
    _call("moe_quant_fp8_128x128_rule", _ptr(w), b, rows, cols, _rule(rule), _ptr(q), _ptr(scale), _stream())
    return q, scale


def pack_w13(q1, s1, q3, s3, q13=None, s13=None):
    """q1, q3 u8 [batch][I][d]; s1, s3 f32 [batch][I/128][d/128] -> W13 in the SwiGLU epilogue layout."""
    b, I, d = q1.shape
    q13 = torch.empty(b, 2 * I, d, dtype=torch.uint8, device=q1.device) if q13 is None else q13
    s13 = torch.empty(b, 2 * I // 128, d // 128, dtype=torch.float32, device=q1.device) if s13 is None else s13
    _call("moe_pack_w13", _ptr(q1), _ptr(s1), _ptr(q3), _ptr(s3), b, I, d, _ptr(q13), _ptr(s13), _stream())
    return q13, s13


def permute(cfg, idx, xq=None, xs=None, workspace=None, out=None, want_counts=False, gather_rows=True):
    """Grouped row order of the (token, expert) pairs; with gather_rows also the
    grouped copy of the quantised tokens xq, xs (otherwise they may be None)."""
    dev = idx.device
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    if gather_rows:
        _need(xq, torch.uint8, "xq", (cfg.T, cfg.d))
        _need(xs, torch.float32, "xs", (cfg.T, cfg.d // 128))
    else:
        xq = xs = None
    rows = cfg.rows
    if out is None:
        out = {
            "offsets": torch.empty(cfg.E + 2, dtype=torch.int32, device=dev),
            "counts": torch.empty(cfg.E, dtype=torch.int32, device=dev) if want_counts else None,
            "sorted_token": torch.empty(cfg.T * cfg.K + cfg.T, dtype=torch.int32, device=dev),
            "row_of": torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev),
            "xq_perm": torch.empty(rows, cfg.d, dtype=torch.uint8, device=dev) if gather_rows else None,
            "xs_perm": torch.empty(rows, cfg.d // 128, dtype=torch.float32, device=dev) if gather_rows else None,
        }
    if workspace is None:
        workspace = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=dev)
    c = config_c(cfg)
    _call("moe_permute", ctypes.byref(c), _ptr(idx), _ptr(xq), _ptr(xs), _ptr(out["offsets"]), _ptr(out["counts"]),
          _ptr(out["sorted_token"]), _ptr(out["row_of"]), _ptr(out["xq_perm"] if gather_rows else None),
          _ptr(out["xs_perm"] if gather_rows else None), _ptr(workspace), workspace.numel(), _stream())
    return out


def permute_noalloc(cfg, idx, xq, xs, out=None, want_counts=False):
    """moe_permute_noalloc: same results as permute(), scratch held inside the library.

    Outputs are allocated here only when the caller passes none; the library
    call itself allocates nothing.
    """
    dev = idx.device
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    _need(xq, torch.uint8, "xq", (cfg.T, cfg.d))
    _need(xs, torch.float32, "xs", (cfg.T, cfg.d // 128))
    rows = cfg.rows
    if out is None:
        out = {
            "offsets": torch.empty(cfg.E + 2, dtype=torch.int32, device=dev),
            "counts": torch.empty(cfg.E, dtype=torch.int32, device=dev) if want_counts else None,
            "sorted_token": torch.empty(cfg.T * cfg.K + cfg.T, dtype=torch.int32, device=dev),
            "row_of": torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev),
            "xq_perm": torch.empty(rows, cfg.d, dtype=torch.uint8, device=dev),
            "xs_perm": torch.empty(rows, cfg.d // 128, dtype=torch.float32, device=dev),
        }
    c = config_c(cfg)
    _call("moe_permute_noalloc", ctypes.byref(c), _ptr(idx), _ptr(xq), _ptr(xs), _ptr(out["offsets"]),
          _ptr(out["counts"]), _ptr(out["sorted_token"]), _ptr(out["row_of"]), _ptr(out["xq_perm"]),
          _ptr(out["xs_perm"]), _stream())
    return out


def grouped_gemm_fp8(offsets, A, sa, B, sb, epilogue=MOE_EPI_BF16, out=None, out_scale=None, last_rows=None,
                     row_index=None, block_scaled=False):
    """offsets i32 [G+1]; A u8 [rows][K]; sa f32 [rows][K/128]; B u8 [G][N][K]; sb f32 [G][N/128][K/128].

    out_scale is the auxiliary output: h scales for the SwiGLU epilogue, or
    the FP32 output of the last group (last_rows rows) for MOE_EPI_BF16_F32_LAST.
    block_scaled: power-of-two scales, run on the block-scaled MMA (moe_grouped_gemm_fp8_mx).
    """
    groups = offsets.numel() - 1
    a_rows, Kdim = A.shape
    rows = a_rows if row_index is None else row_index.numel()
    N = B.shape[1]
    _need(offsets, torch.int32, "offsets")
    _need(A, torch.uint8, "A")
    _need(sa, torch.float32, "sa", (a_rows, Kdim // 128))
    if row_index is not None:
        _need(row_index, torch.int32, "row_index")
    _need(B, torch.uint8, "B", (groups, N, Kdim))
    _need(sb, torch.float32, "sb", (groups, N // 128, Kdim // 128))
    if epilogue == MOE_EPI_BF16:
        out = torch.empty(rows, N, dtype=torch.bfloat16, device=A.device) if out is None else out
    elif epilogue == MOE_EPI_BF16_F32_LAST:
        out = torch.empty(rows, N, dtype=torch.bfloat16, device=A.device) if out is None else out
        if out_scale is None:
            out_scale = torch.empty(last_rows, N, dtype=torch.float32, device=A.device)
    elif epilogue in (MOE_EPI_F32, MOE_EPI_GATEUP_F32):
        out = torch.empty(rows, N, dtype=torch.float32, device=A.device) if out is None else out
    else:
        out = torch.empty(rows, N // 2, dtype=torch.uint8, device=A.device) if out is None else out
        out_scale = (torch.empty(rows, N // 256, dtype=torch.float32, device=A.device)
                     if out_scale is None else out_scale)
    if block_scaled:
        if row_index is not None:
            raise ValueError("the block-scaled GEMM reads A in grouped row order (no row_index)")
        _call("moe_grouped_gemm_fp8_mx", groups, _ptr(offsets), rows, N, Kdim, _ptr(A), _ptr(sa), _ptr(B), _ptr(sb),
              epilogue, _ptr(out), _ptr(out_scale), _stream())
    elif row_index is None:
        _call("moe_grouped_gemm_fp8", groups, _ptr(offsets), rows, N, Kdim, _ptr(A), _ptr(sa), _ptr(B), _ptr(sb),
              epilogue, _ptr(out), _ptr(out_scale), _stream())
    else:
        _call("moe_grouped_gemm_fp8_gather", groups, _ptr(offsets), rows, N, Kdim, _ptr(A), _ptr(sa), a_rows,
              _ptr(row_index), _ptr(B), _ptr(sb), epilogue, _ptr(out), _ptr(out_scale), _stream())
    return out, out_scale


def balance_loss(cfg, idx, workspace, seq_len, alpha, logit_offset=None, stats=True):
    """Per-sequence L_Bal after moe_route on `workspace`; returns (loss [T/seq_len], f, P) with
    f, P [T/seq_len][E] (None unless stats)."""
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    nseq = cfg.T // seq_len
    dev = idx.device
    loss = torch.empty(nseq, dtype=torch.float32, device=dev)
    f = torch.empty(nseq, cfg.E, dtype=torch.float32, device=dev) if stats else None
    P = torch.empty(nseq, cfg.E, dtype=torch.float32, device=dev) if stats else None
    c = config_c(cfg)
    _call("moe_balance_loss", ctypes.byref(c), _ptr(logit_offset), _ptr(idx), seq_len, alpha, _ptr(f), _ptr(P),
          _ptr(loss), _ptr(workspace), workspace.numel(), _stream())
    return loss, f, P


def combine(cfg, routed_out, shared_out, row_of, gate, residual=None, y=None):
    """routed_out bf16 [T*K][d], shared_out f32 [T][d] -> y bf16 [T][d]."""
    _need(routed_out, torch.bfloat16, "routed_out", (cfg.T * cfg.K, cfg.d))
    _need(shared_out, torch.float32, "shared_out", (cfg.T, cfg.d))
    _need(row_of, torch.int32, "row_of", (cfg.T, cfg.K))
    _need(gate, torch.float32, "topk_gate", (cfg.T, cfg.K))
    y = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=row_of.device) if y is None else y
    c = config_c(cfg)
    _call("moe_combine", ctypes.byref(c), _ptr(routed_out), _ptr(shared_out), _ptr(row_of), _ptr(gate),
          _ptr(residual), _ptr(y), _stream())
    return y


def bias_update(E, T, K, counts, gamma, bias):
    _need(counts, torch.int32, "counts", (E,))
    _need(bias, torch.float32, "bias", (E,))
    _call("moe_bias_update", E, T, K, _ptr(counts), ctypes.c_float(gamma), _ptr(bias), _stream())
    return bias


# ------------------------------------------------------------------ backward ----
def transpose_fp8_blocks(q, scale, qT=None, scaleT=None, offset: int = 0):
    """q u8 [batch][rows][cols], scale f32 [batch][rows/128][cols/128] -> transposed blocks.

    qT u8 [batch][colsT][ldT] and scaleT f32 [batch][colsT/128][ldT/128] (allocated
    [batch][cols][rows] when None); the source's rows land in columns offset ..
    offset + rows - 1 of qT (offset a multiple of 128), so two matrices can share
    qT side by side; rows cols .. colsT-1 of each matrix are left as they are.
    """
    _need(q, torch.uint8, "q")
    b, rows, cols = q.shape
    _need(scale, torch.float32, "scale", (b, rows // 128, cols // 128))
    if qT is None:
        qT = torch.empty(b, cols, rows, dtype=torch.uint8, device=q.device)
        scaleT = torch.empty(b, cols // 128, rows // 128, dtype=torch.float32, device=q.device)
    _need(qT, torch.uint8, "qT")
    _need(scaleT, torch.float32, "scaleT")
    colsT, ldT = qT.shape[1], qT.shape[2]
    if qT.shape[0] != b or colsT < cols or offset % 128 or offset + rows > ldT or \
            tuple(scaleT.shape) != (b, colsT // 128, ldT // 128):
        raise ValueError("qT / scaleT do not fit the transposed blocks")
    _call("moe_transpose_fp8_blocks", _ptr(q), _ptr(scale), b, rows, cols, ctypes.c_void_p(qT.data_ptr() + offset),
          ctypes.c_void_p(scaleT.data_ptr() + 4 * (offset // 128)), ldT, colsT, _stream())
    return qT, scaleT


def combine_backward(cfg, dy, routed_out, row_of, gate, dOq, dOs, row_gate, dgate, rule="fp32"):
    _need(dy, torch.bfloat16, "dy", (cfg.T, cfg.d))
    _need(routed_out, torch.bfloat16, "routed_out")
    if routed_out.shape[0] < cfg.T * cfg.K or routed_out.shape[1] != cfg.d:
        raise ValueError("routed_out: expected at least T*K rows of d columns")
    _need(row_of, torch.int32, "row_of", (cfg.T, cfg.K))
    _need(gate, torch.float32, "topk_gate", (cfg.T, cfg.K))
    _need(dOq, torch.uint8, "dOq", (cfg.rows, cfg.d))
    _need(dOs, torch.float32, "dOs", (cfg.rows, cfg.d // 128))
    _need(row_gate, torch.float32, "row_gate", (cfg.rows,))
    _need(dgate, torch.float32, "dgate", (cfg.T, cfg.K))
    c = config_c(cfg)
    _call("moe_combine_backward", ctypes.byref(c), _ptr(dy), _ptr(routed_out), _ptr(row_of), _ptr(gate), _rule(rule),
          _ptr(dOq), _ptr(dOs), _ptr(row_gate), _ptr(dgate), _stream())


def route_backward(cfg, idx, dgate, workspace, dz, logit_offset=None):
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    _need(dgate, torch.float32, "dgate", (cfg.T, cfg.K))
    _need(dz, torch.float32, "dz", (cfg.T, cfg.K))
    c = config_c(cfg)
    _call("moe_route_backward", ctypes.byref(c), _ptr(logit_offset), _ptr(idx), _ptr(dgate), _ptr(dz),
          _ptr(workspace), workspace.numel(), _stream())


def router_wgrad(cfg, x, offsets, sorted_token, row_of, dz, dWr):
    _need(x, torch.bfloat16, "x", (cfg.T, cfg.d))
    _need(offsets, torch.int32, "offsets")
    _need(sorted_token, torch.int32, "sorted_token")
    _need(row_of, torch.int32, "row_of", (cfg.T, cfg.K))
    _need(dz, torch.float32, "dz", (cfg.T, cfg.K))
    _need(dWr, torch.float32, "dWr", (cfg.E, cfg.d))
    c = config_c(cfg)
    _call("moe_router_wgrad", ctypes.byref(c), _ptr(x), _ptr(offsets), _ptr(sorted_token), _ptr(row_of), _ptr(dz),
          _ptr(dWr), _stream())


def swiglu_backward(ab, dh, dab_q, dab_s, rule="fp32"):
    """ab f32 [rows][2I] (a|b in the gate/up tile layout; overwritten by dA|dB), dh f32
    [rows][>= I] (the first I columns are read)."""
    _need(ab, torch.float32, "ab")
    rows, I2 = ab.shape
    _need(dh, torch.float32, "dh")
    if dh.shape[0] != rows or dh.shape[1] < I2 // 2:
        raise ValueError("dh: expected [rows][>= I]")
    _need(dab_q, torch.uint8, "dab_q", (rows, I2))
    _need(dab_s, torch.float32, "dab_s", (rows, I2 // 128))
    _call("moe_swiglu_backward", rows, I2 // 2, _ptr(ab), _ptr(dh), dh.shape[1], _rule(rule), _ptr(dab_q),
          _ptr(dab_s), _stream())


def dx_combine(cfg, dx_routed, dx_shared, row_of, idx, dz, Wr, dx):
    _need(dx_routed, torch.bfloat16, "dx_routed")
    if dx_routed.shape[0] < cfg.T * cfg.K or dx_routed.shape[1] != cfg.d:
        raise ValueError("dx_routed: expected at least T*K rows of d columns")
    _need(dx_shared, torch.float32, "dx_shared", (cfg.T, cfg.d))
    _need(row_of, torch.int32, "row_of", (cfg.T, cfg.K))
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    _need(dz, torch.float32, "dz", (cfg.T, cfg.K))
    _need(Wr, torch.float32, "Wr", (cfg.E, cfg.d))
    _need(dx, torch.bfloat16, "dx", (cfg.T, cfg.d))
    c = config_c(cfg)
    _call("moe_dx_combine", ctypes.byref(c), _ptr(dx_routed), _ptr(dx_shared), _ptr(row_of), _ptr(idx), _ptr(dz),
          _ptr(Wr), _ptr(dx), _stream())


def q1_width(groups: int, rows: int) -> int:
    """Columns a 128x1 grouped operand may need: 128 * (ceil(rows/128) + groups)."""
    return 128 * ((rows + 127) // 128 + groups)


def _q1_out(cols, width, dev, qT, sT):
    qT = torch.empty(cols, width, dtype=torch.uint8, device=dev) if qT is None else qT
    sT = torch.empty(width // 128, cols, dtype=torch.float32, device=dev) if sT is None else sT
    _need(qT, torch.uint8, "qT")
    _need(sT, torch.float32, "sT")
    if qT.shape[0] != cols or sT.shape[1] != cols or sT.shape[0] * 128 < qT.shape[1]:
        raise ValueError("qT [cols][width] and sT [width/128][cols] do not match")
    return qT, sT


def quant_128x1(offsets, rows, cols, rule="fp32", qT=None, sT=None, *, f32=None, fp8=None, bf16_rows=None):
    """128x1 grouped quantisation of one source (exactly one of):
      f32=v [rows][cols]; fp8=(q [rows][cols], s [rows][cols/128]);
      bf16_rows=(x [X][cols], row_map i32 [rows], row_mult f32 [rows] or None).
    Returns (qT u8 [cols][width], sT f32 [width/128][cols])."""
    _need(offsets, torch.int32, "offsets")
    groups = offsets.numel() - 1
    dev = offsets.device
    qT, sT = _q1_out(cols, q1_width(groups, rows) if qT is None else qT.shape[1], dev, qT, sT)
    tail = (groups, _ptr(offsets), rows, cols, _rule(rule), _ptr(qT), qT.shape[1], _ptr(sT), _stream())
    if f32 is not None:
        _need(f32, torch.float32, "v")
        _call("moe_quant_fp8_128x1_f32", _ptr(f32), f32.shape[1], *tail)
    elif fp8 is not None:
        q, s = fp8
        _need(q, torch.uint8, "q")
        _need(s, torch.float32, "scale", (q.shape[0], q.shape[1] // 128))
        _call("moe_quant_fp8_128x1_fp8", _ptr(q), _ptr(s), q.shape[1], *tail)
    else:
        x, row_map, row_mult = bf16_rows
        _need(x, torch.bfloat16, "x")
        _need(row_map, torch.int32, "row_map")
        if row_mult is not None:
            _need(row_mult, torch.float32, "row_mult")
        _call("moe_quant_fp8_128x1_bf16_rows", _ptr(x), x.shape[0], x.shape[1], _ptr(row_map), _ptr(row_mult), *tail)
    return qT, sT


def grouped_wgrad_fp8(offsets, rows, AT, saT, BT, sbT, out=None):
    """out[g] = AT_g . BT_g^T over group g's 128-row tiles (see moe_grouped_wgrad_fp8)."""
    _need(offsets, torch.int32, "offsets")
    groups = offsets.numel() - 1
    _need(AT, torch.uint8, "AT")
    _need(BT, torch.uint8, "BT")
    M, width = AT.shape
    N = BT.shape[0]
    if BT.shape[1] != width:
        raise ValueError("AT and BT must have the same width")
    _need(saT, torch.float32, "saT")
    _need(sbT, torch.float32, "sbT")
    if saT.shape[1] != M or sbT.shape[1] != N or saT.shape[0] * 128 < width or sbT.shape[0] * 128 < width:
        raise ValueError("scale shapes do not match the operands")
    out = torch.empty(groups, M, N, dtype=torch.float32, device=AT.device) if out is None else out
    _need(out, torch.float32, "out", (groups, M, N))
    _call("moe_grouped_wgrad_fp8", groups, _ptr(offsets), rows, width, M, N, _ptr(AT), _ptr(saT), _ptr(BT), _ptr(sbT),
          _ptr(out), _stream())
    return out


# ------------------------------------------------------------------ expert parallel ----
def ep_row_bytes(d: int, K: int) -> int:
    return int(load().moe_ep_row_bytes(d, K))


def ep_workspace_size(cfg, R: int, rows: int) -> int:
    c = config_c(cfg)
    return int(load().moe_ep_workspace_size(ctypes.byref(c), R, rows))


def ep_dispatch(cfg, R, idx, gate, xq, xs, workspace=None):
    """moe_ep_dispatch: packed send rows ordered by (destination rank, token). Returns a dict
    with send_counts [R], send_offsets [R+1], send_row_of [T][K], send_token and send_buf
    (capacity T*min(K,R) rows; the first send_offsets[R] are written)."""
    dev = idx.device
    _need(idx, torch.int32, "topk_idx", (cfg.T, cfg.K))
    _need(gate, torch.float32, "topk_gate", (cfg.T, cfg.K))
    _need(xq, torch.uint8, "xq", (cfg.T, cfg.d))
    _need(xs, torch.float32, "xs", (cfg.T, cfg.d // 128))
    cap = cfg.T * min(cfg.K, R)
    out = {"send_counts": torch.empty(R, dtype=torch.int32, device=dev),
           "send_offsets": torch.empty(R + 1, dtype=torch.int32, device=dev),
           "send_row_of": torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev),
           "send_token": torch.empty(cap, dtype=torch.int32, device=dev),
           "send_buf": torch.empty(cap, ep_row_bytes(cfg.d, cfg.K), dtype=torch.uint8, device=dev)}
    if workspace is None:
        workspace = torch.empty(max(ep_workspace_size(cfg, R, cfg.T), 16), dtype=torch.uint8, device=dev)
    c = config_c(cfg)
    _call("moe_ep_dispatch", ctypes.byref(c), R, _ptr(idx), _ptr(gate), _ptr(xq), _ptr(xs), _ptr(out["send_counts"]),
          _ptr(out["send_offsets"]), _ptr(out["send_row_of"]), _ptr(out["send_token"]), _ptr(out["send_buf"]),
          _ptr(workspace), workspace.numel(), _stream())
    return out


def ep_receive(cfg, R, rank, recv_buf, workspace=None, want_counts=False):
    """moe_ep_receive on packed rows recv_buf u8 [n][row_bytes]: this rank's pairs grouped by
    local expert, with their codes and scales gathered (capacity n*K rows)."""
    n = recv_buf.shape[0]
    dev = recv_buf.device
    _need(recv_buf, torch.uint8, "recv_buf", (n, ep_row_bytes(cfg.d, cfg.K)))
    nl = cfg.E // R
    cap = max(n * cfg.K, 1)
    out = {"local_offsets": torch.empty(nl + 1, dtype=torch.int32, device=dev),
           "local_counts": torch.empty(nl, dtype=torch.int32, device=dev) if want_counts else None,
           "sorted_row": torch.empty(cap, dtype=torch.int32, device=dev),
           "row_of": torch.empty(max(n, 1), cfg.K, dtype=torch.int32, device=dev),
           "xq_local": torch.empty(cap, cfg.d, dtype=torch.uint8, device=dev),
           "xs_local": torch.empty(cap, cfg.d // 128, dtype=torch.float32, device=dev)}
    if workspace is None:
        workspace = torch.empty(max(ep_workspace_size(cfg, R, n), 16), dtype=torch.uint8, device=dev)
    c = config_c(cfg)
    _call("moe_ep_receive", ctypes.byref(c), R, rank, n, _ptr(recv_buf) if n else None, _ptr(out["local_offsets"]),
          _ptr(out["local_counts"]), _ptr(out["sorted_row"]), _ptr(out["row_of"]), _ptr(out["xq_local"]),
          _ptr(out["xs_local"]), _ptr(workspace), workspace.numel(), _stream())
    return out


def ep_partial(cfg, recv_buf, row_of, routed_out, partial=None):
    """moe_ep_partial: per received row the gate-weighted sum of this rank's expert outputs (FP32)."""
    n = recv_buf.shape[0]
    _need(routed_out, torch.bfloat16, "routed_out")
    partial = torch.empty(n, cfg.d, dtype=torch.float32, device=recv_buf.device) if partial is None else partial
    c = config_c(cfg)
    _call("moe_ep_partial", ctypes.byref(c), n, _ptr(recv_buf), _ptr(row_of), _ptr(routed_out), routed_out.shape[0],
          _ptr(partial), _stream())
    return partial


def ep_combine(cfg, shared_out, returned, send_row_of, residual=None, y=None):
    """moe_ep_combine: y = shared + the partial rows returned for each token (+ residual), bf16."""
    _need(shared_out, torch.float32, "shared_out", (cfg.T, cfg.d))
    _need(send_row_of, torch.int32, "send_row_of", (cfg.T, cfg.K))
    _need(returned, torch.float32, "returned")
    y = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=shared_out.device) if y is None else y
    c = config_c(cfg)
    _call("moe_ep_combine", ctypes.byref(c), _ptr(shared_out), _ptr(returned) if returned.numel() else None,
          returned.shape[0], _ptr(send_row_of), _ptr(residual), _ptr(y), _stream())
    return y
