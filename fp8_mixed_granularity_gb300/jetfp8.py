"""Thin Python binding of libjetfp8.so (the C ABI in include/jetfp8.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks dtype/shape/contiguity, passes raw device pointers and
the current CUDA stream to the C entry point of the same name, and raises
JetFP8Error on a non-OK status.  No arithmetic of the method happens here and
there is no fallback: if the library is missing, loading it raises.

Scale tensors use the library's group-index-major layout: the scales of an
[R, C] tensor quantised in 1×128 row groups are a float32 tensor
[C/128, roundup(R, 4)]; `scale_shape()` gives that shape.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libjetfp8.so")

JETFP8_OK = 0
OUT_BF16 = 0
OUT_FP32 = 1

_STATUS = {0: "JETFP8_OK", 1: "JETFP8_ERR_INVALID_ARG", 2: "JETFP8_ERR_UNSUPPORTED_SHAPE",
           3: "JETFP8_ERR_MISALIGNED", 4: "JETFP8_ERR_CUDA", 5: "JETFP8_ERR_TIMEOUT",
           6: "JETFP8_ERR_UNSUPPORTED"}

# name -> argument types (all entry points return jetfp8_status as int)
_P, _I64, _F32, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
SIGNATURES = {
    "jetfp8_quant_act_1x128": [_P, _I64, _I64, _P, _P, _P],
    "jetfp8_quant_weight_128x128": [_P, _I64, _I64, _P, _P, _P, _P],
    "jetfp8_requant_rowgrp_to_colgrp": [_P, _P, _I64, _I64, _P, _P, _P],
    "jetfp8_quant_grad_dual": [_P, _I64, _I64, _P, _P, _P, _P, _P],
    "jetfp8_rmsnorm_quant": [_P, _P, _F32, _I64, _I64, _P, _P, _P, _P, _P],
    "jetfp8_gemm_fprop": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _INT, _P],
    "jetfp8_gemm_dgrad": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _INT, _P],
    "jetfp8_gemm_wgrad": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _INT, _P],
    "jetfp8_gemm_wgrad_grouped": [_INT, _P, _P, _P, _P, _I64, _P, _P, _P, _INT, _P],
    "jetfp8_quant_weight_grouped": [_INT, _P, _P, _P, _P, _P, _P, _P],
    "jetfp8_test_gemm_fprop_drop_block": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _INT, _P],
    "jetfp8_gemm_fprop_quant": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "jetfp8_gemm_dgrad_quant": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "jetfp8_rmsnorm_bwd": [_P, _P, _P, _P, _I64, _I64, _P, _P, _P, ctypes.c_size_t, _P],
    "jetfp8_rmsnorm_bwd_noalloc": [_P, _P, _P, _P, _I64, _I64, _P, _P, _P],
    "jetfp8_swiglu_quant": [_P, _I64, _I64, _P, _P, _P, _P],
    "jetfp8_swiglu_bwd": [_P, _P, _I64, _I64, _P, _P],
    "jetfp8_get_last_device_error": [_P],
    "jetfp8_test_set_gemm_path": [_INT],
    "jetfp8_quant_nvfp4": [_P, _I64, _I64, _P, _P, _P, _P],
    "jetfp8_gemm_fprop_nvfp4": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P],
}


class JetFP8Error(RuntimeError):
    pass


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libjetfp8.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise JetFP8Error(f"{path} not found: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
        lib = ctypes.CDLL(path)
        for name, argtypes in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = ctypes.c_int
        lib.jetfp8_status_string.argtypes = [ctypes.c_int]
        lib.jetfp8_status_string.restype = ctypes.c_char_p
        lib.jetfp8_rmsnorm_bwd_workspace_bytes.argtypes = [_I64, _I64]
        lib.jetfp8_rmsnorm_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.jetfp8_nvfp4_scale_bytes.argtypes = [_I64, _I64]
        lib.jetfp8_nvfp4_scale_bytes.restype = ctypes.c_size_t
        _lib = lib
    return _lib


def _check(status: int, name: str) -> None:
    if status != JETFP8_OK:
        raise JetFP8Error(f"{name} returned {_STATUS.get(status, status)}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, shape=None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise JetFP8Error(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise JetFP8Error(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise JetFP8Error(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise JetFP8Error(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def round_up4(n: int) -> int:
    return (n + 3) // 4 * 4


def scale_shape(rows: int, cols: int) -> tuple[int, int]:
    """Scale tensor shape for an [rows, cols] tensor in 1×128 row groups."""
    return (cols // 128, round_up4(rows))


_U8, _F, _BF = torch.uint8, torch.float32, torch.bfloat16


def jetfp8_quant_act_1x128(x, q, s, stream=None):
    M, K = x.shape
    _check(load_library().jetfp8_quant_act_1x128(
        _ptr(x, _BF, None, "x"), M, K, _ptr(q, _U8, (M, K), "q"), _ptr(s, _F, scale_shape(M, K), "s"),
        _stream(stream)), "jetfp8_quant_act_1x128")


def jetfp8_quant_weight_128x128(w, q, s, qT=None, stream=None):
    N, K = w.shape
    _check(load_library().jetfp8_quant_weight_128x128(
        _ptr(w, _BF, None, "w"), N, K, _ptr(q, _U8, (N, K), "q"), _ptr(s, _F, (N // 128, K // 128), "s"),
        _ptr(qT, _U8, (K, N), "qT"), _stream(stream)), "jetfp8_quant_weight_128x128")


def jetfp8_requant_rowgrp_to_colgrp(q, s, qT, sT, stream=None):
    M, K = q.shape
    _check(load_library().jetfp8_requant_rowgrp_to_colgrp(
        _ptr(q, _U8, None, "q"), _ptr(s, _F, scale_shape(M, K), "s"), M, K,
        _ptr(qT, _U8, (K, M), "qT"), _ptr(sT, _F, scale_shape(K, M), "sT"), _stream(stream)),
        "jetfp8_requant_rowgrp_to_colgrp")


def jetfp8_quant_grad_dual(dy, q_row, s_row, qT_col=None, sT_col=None, stream=None):
    M, N = dy.shape
    _check(load_library().jetfp8_quant_grad_dual(
        _ptr(dy, _BF, None, "dy"), M, N, _ptr(q_row, _U8, (M, N), "q_row"),
        _ptr(s_row, _F, scale_shape(M, N), "s_row"), _ptr(qT_col, _U8, (N, M), "qT_col"),
        _ptr(sT_col, _F, None if sT_col is None else scale_shape(N, M), "sT_col"), _stream(stream)),
        "jetfp8_quant_grad_dual")


def jetfp8_rmsnorm_quant(x, gamma, eps, q, s, rstd, y=None, stream=None):
    M, H = x.shape
    _check(load_library().jetfp8_rmsnorm_quant(
        _ptr(x, _BF, None, "x"), _ptr(gamma, _BF, (H,), "gamma"), float(eps), M, H,
        _ptr(q, _U8, (M, H), "q"), _ptr(s, _F, scale_shape(M, H), "s"), _ptr(rstd, _F, (M,), "rstd"),
        _ptr(y, _BF, (M, H), "y"), _stream(stream)), "jetfp8_rmsnorm_quant")


def _out_dt(out: torch.Tensor) -> int:
    if out.dtype == _BF:
        return OUT_BF16
    if out.dtype == _F:
        return OUT_FP32
    raise JetFP8Error("output must be bfloat16 or float32")


def jetfp8_gemm_fprop(xq, sx, wq, sw, y, stream=None):
    M, K = xq.shape
    N = wq.shape[0]
    _check(load_library().jetfp8_gemm_fprop(
        _ptr(xq, _U8, None, "xq"), _ptr(sx, _F, scale_shape(M, K), "sx"), _ptr(wq, _U8, (N, K), "wq"),
        _ptr(sw, _F, (N // 128, K // 128), "sw"), M, N, K, _ptr(y, None, (M, N), "y"), _out_dt(y),
        _stream(stream)), "jetfp8_gemm_fprop")


def jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx, stream=None):
    M, N = dyq.shape
    K = wqT.shape[0]
    _check(load_library().jetfp8_gemm_dgrad(
        _ptr(dyq, _U8, None, "dyq"), _ptr(sdy, _F, scale_shape(M, N), "sdy"), _ptr(wqT, _U8, (K, N), "wqT"),
        _ptr(sw, _F, (N // 128, K // 128), "sw"), M, N, K, _ptr(dx, None, (M, K), "dx"), _out_dt(dx),
        _stream(stream)), "jetfp8_gemm_dgrad")


def jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw, stream=None):
    N, M = dyqT.shape
    K = xqT.shape[0]
    _check(load_library().jetfp8_gemm_wgrad(
        _ptr(dyqT, _U8, None, "dyqT"), _ptr(sdyT, _F, scale_shape(N, M), "sdyT"),
        _ptr(xqT, _U8, (K, M), "xqT"), _ptr(sxT, _F, scale_shape(K, M), "sxT"), M, N, K,
        _ptr(dw, None, (N, K), "dw"), _out_dt(dw), _stream(stream)), "jetfp8_gemm_wgrad")


def jetfp8_test_gemm_fprop_drop_block(xq, sx, wq, sw, y, drop_kb, stream=None):
    """Failure-path test hook: FProp whose producer never loads block `drop_kb`;
    the bounded wait runs out and jetfp8_get_last_device_error reports it."""
    M, K = xq.shape
    N = wq.shape[0]
    _check(load_library().jetfp8_test_gemm_fprop_drop_block(
        _ptr(xq, _U8, None, "xq"), _ptr(sx, _F, scale_shape(M, K), "sx"), _ptr(wq, _U8, (N, K), "wq"),
        _ptr(sw, _F, (N // 128, K // 128), "sw"), M, N, K, _ptr(y, _BF, (M, N), "y"), int(drop_kb),
        _stream(stream)), "jetfp8_test_gemm_fprop_drop_block")


MAX_GROUP = 4


def jetfp8_gemm_wgrad_grouped(problems, stream=None):
    """WGrads of up to MAX_GROUP linears sharing the token count M in one launch.
    `problems`: a list of (dyqT, sdyT, xqT, sxT, dw) as for jetfp8_gemm_wgrad;
    every dw has the same dtype."""
    n = len(problems)
    if not 1 <= n <= MAX_GROUP:
        raise JetFP8Error(f"jetfp8_gemm_wgrad_grouped: {n} problems (1..{MAX_GROUP})")
    M = problems[0][0].shape[1]
    cols = [[] for _ in range(5)]
    Ns, Ks = [], []
    for dyqT, sdyT, xqT, sxT, dw in problems:
        N, K = dyqT.shape[0], xqT.shape[0]
        if dyqT.shape[1] != M or dw.dtype != problems[0][4].dtype:
            raise JetFP8Error("jetfp8_gemm_wgrad_grouped: problems differ in M or output dtype")
        cols[0].append(_ptr(dyqT, _U8, (N, M), "dyqT"))
        cols[1].append(_ptr(sdyT, _F, scale_shape(N, M), "sdyT"))
        cols[2].append(_ptr(xqT, _U8, (K, M), "xqT"))
        cols[3].append(_ptr(sxT, _F, scale_shape(K, M), "sxT"))
        cols[4].append(_ptr(dw, None, (N, K), "dw"))
        Ns.append(N)
        Ks.append(K)
    arrs = [(ctypes.c_void_p * n)(*c) for c in cols]
    _check(load_library().jetfp8_gemm_wgrad_grouped(
        n, arrs[0], arrs[1], arrs[2], arrs[3], M, (ctypes.c_int64 * n)(*Ns), (ctypes.c_int64 * n)(*Ks),
        arrs[4], _out_dt(problems[0][4]), _stream(stream)), "jetfp8_gemm_wgrad_grouped")


def jetfp8_quant_weight_grouped(problems, stream=None):
    """Q2 of up to MAX_GROUP weights in one launch.  `problems`: a list of
    (w, q, s, qT) as for jetfp8_quant_weight_128x128 (qT may be None)."""
    n = len(problems)
    if not 1 <= n <= MAX_GROUP:
        raise JetFP8Error(f"jetfp8_quant_weight_grouped: {n} problems (1..{MAX_GROUP})")
    cols = [[] for _ in range(4)]
    Ns, Ks = [], []
    for w, q, s, qT in problems:
        N, K = w.shape
        cols[0].append(_ptr(w, _BF, (N, K), "w"))
        cols[1].append(_ptr(q, _U8, (N, K), "q"))
        cols[2].append(_ptr(s, _F, (N // 128, K // 128), "s"))
        cols[3].append(_ptr(qT, _U8, (K, N), "qT"))
        Ns.append(N)
        Ks.append(K)
    arrs = [(ctypes.c_void_p * n)(*c) for c in cols]
    _check(load_library().jetfp8_quant_weight_grouped(
        n, arrs[0], (ctypes.c_int64 * n)(*Ns), (ctypes.c_int64 * n)(*Ks), arrs[1], arrs[2], arrs[3],
        _stream(stream)), "jetfp8_quant_weight_grouped")


def jetfp8_gemm_fprop_quant(xq, sx, wq, sw, yq, ys, y=None, stream=None):
    """FProp with the 1×128 quantiser of its bf16 output fused in (y optional)."""
    M, K = xq.shape
    N = wq.shape[0]
    _check(load_library().jetfp8_gemm_fprop_quant(
        _ptr(xq, _U8, None, "xq"), _ptr(sx, _F, scale_shape(M, K), "sx"), _ptr(wq, _U8, (N, K), "wq"),
        _ptr(sw, _F, (N // 128, K // 128), "sw"), M, N, K, _ptr(y, _BF, (M, N), "y"),
        _ptr(yq, _U8, (M, N), "yq"), _ptr(ys, _F, scale_shape(M, N), "ys"), _stream(stream)),
        "jetfp8_gemm_fprop_quant")


def jetfp8_gemm_dgrad_quant(dyq, sdy, wqT, sw, dxq, dxs, dx=None, stream=None):
    """DGrad with the 1×128 quantiser of its bf16 output fused in (dx optional)."""
    M, N = dyq.shape
    K = wqT.shape[0]
    _check(load_library().jetfp8_gemm_dgrad_quant(
        _ptr(dyq, _U8, None, "dyq"), _ptr(sdy, _F, scale_shape(M, N), "sdy"), _ptr(wqT, _U8, (K, N), "wqT"),
        _ptr(sw, _F, (N // 128, K // 128), "sw"), M, N, K, _ptr(dx, _BF, (M, K), "dx"),
        _ptr(dxq, _U8, (M, K), "dxq"), _ptr(dxs, _F, scale_shape(M, K), "dxs"), _stream(stream)),
        "jetfp8_gemm_dgrad_quant")


def jetfp8_rmsnorm_bwd_workspace_bytes(M: int, H: int) -> int:
    return int(load_library().jetfp8_rmsnorm_bwd_workspace_bytes(M, H))


def jetfp8_rmsnorm_bwd(x, gamma, rstd, dy, dx, dgamma, workspace, stream=None):
    """RMSNorm backward; `workspace` is a device tensor of at least
    jetfp8_rmsnorm_bwd_workspace_bytes(M, H) bytes (its contents are overwritten)."""
    M, H = x.shape
    _check(load_library().jetfp8_rmsnorm_bwd(
        _ptr(x, _BF, None, "x"), _ptr(gamma, _BF, (H,), "gamma"), _ptr(rstd, _F, (M,), "rstd"),
        _ptr(dy, _BF, (M, H), "dy"), M, H, _ptr(dx, _BF, (M, H), "dx"), _ptr(dgamma, _F, (H,), "dgamma"),
        _ptr(workspace, None, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "jetfp8_rmsnorm_bwd")


def jetfp8_rmsnorm_bwd_noalloc(x, gamma, rstd, dy, dx, dgamma, stream=None):
    """RMSNorm backward using the library's fixed scratch (no workspace; calls
    that overlap in time race on that scratch)."""
    M, H = x.shape
    _check(load_library().jetfp8_rmsnorm_bwd_noalloc(
        _ptr(x, _BF, None, "x"), _ptr(gamma, _BF, (H,), "gamma"), _ptr(rstd, _F, (M,), "rstd"),
        _ptr(dy, _BF, (M, H), "dy"), M, H, _ptr(dx, _BF, (M, H), "dx"), _ptr(dgamma, _F, (H,), "dgamma"),
        _stream(stream)), "jetfp8_rmsnorm_bwd_noalloc")


def jetfp8_swiglu_quant(gu, q, s, h=None, stream=None):
    M, I2 = gu.shape
    I = I2 // 2
    _check(load_library().jetfp8_swiglu_quant(
        _ptr(gu, _BF, None, "gu"), M, I, _ptr(q, _U8, (M, I), "q"), _ptr(s, _F, scale_shape(M, I), "s"),
        _ptr(h, _BF, (M, I), "h"), _stream(stream)), "jetfp8_swiglu_quant")


def jetfp8_swiglu_bwd(gu, dh, dgu, stream=None):
    M, I2 = gu.shape
    I = I2 // 2
    _check(load_library().jetfp8_swiglu_bwd(
        _ptr(gu, _BF, None, "gu"), _ptr(dh, _BF, (M, I), "dh"), M, I, _ptr(dgu, _BF, (M, I2), "dgu"),
        _stream(stream)), "jetfp8_swiglu_bwd")


def jetfp8_test_set_gemm_path(mode: int):
    """Kernel choice of later GEMM launches: 0 automatic, 1 single-CTA tiles,
    2 CTA-pair tiles wherever allowed (results are identical either way)."""
    _check(load_library().jetfp8_test_set_gemm_path(int(mode)), "jetfp8_test_set_gemm_path")


def jetfp8_get_last_device_error(stream=None):
    _check(load_library().jetfp8_get_last_device_error(_stream(stream)), "jetfp8_get_last_device_error")


# ---------------------------------------------------------------------------
# Allocation helpers (torch.empty on the device; no computation)
# ---------------------------------------------------------------------------
def jetfp8_nvfp4_scale_bytes(R: int, K: int) -> int:
    return int(load_library().jetfp8_nvfp4_scale_bytes(R, K))


def jetfp8_quant_nvfp4(x, q, sf, g, stream=None):
    """FP4 variant: bf16 rows x [R, K] -> codes q uint8 [R, K/2], block scales sf
    uint8 [jetfp8_nvfp4_scale_bytes(R, K)] (blocked layout), row scales g float32 [R]."""
    R, K = x.shape
    _check(load_library().jetfp8_quant_nvfp4(
        _ptr(x, _BF, None, "x"), R, K, _ptr(q, _U8, (R, K // 2), "q"),
        _ptr(sf, _U8, (jetfp8_nvfp4_scale_bytes(R, K),), "sf"), _ptr(g, _F, (R,), "g"), _stream(stream)),
        "jetfp8_quant_nvfp4")


def jetfp8_gemm_fprop_nvfp4(xq, xsf, gx, wq, wsf, gw, y, stream=None):
    """FP4 variant FProp: y bf16 [M, N] from jetfp8_quant_nvfp4 of X [M, K] and W [N, K]."""
    M, K2 = xq.shape
    N = wq.shape[0]
    K = 2 * K2
    _check(load_library().jetfp8_gemm_fprop_nvfp4(
        _ptr(xq, _U8, None, "xq"), _ptr(xsf, _U8, (jetfp8_nvfp4_scale_bytes(M, K),), "xsf"),
        _ptr(gx, _F, (M,), "gx"), _ptr(wq, _U8, (N, K2), "wq"),
        _ptr(wsf, _U8, (jetfp8_nvfp4_scale_bytes(N, K),), "wsf"), _ptr(gw, _F, (N,), "gw"), M, N, K,
        _ptr(y, _BF, (M, N), "y"), _stream(stream)), "jetfp8_gemm_fprop_nvfp4")


def empty_nvfp4(rows: int, cols: int, device) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(codes uint8 [rows, cols/2], block scales uint8 [scale bytes], row scales float32 [rows])"""
    return (torch.empty(rows, cols // 2, dtype=torch.uint8, device=device),
            torch.empty(jetfp8_nvfp4_scale_bytes(rows, cols), dtype=torch.uint8, device=device),
            torch.empty(rows, dtype=torch.float32, device=device))


def empty_rowgroup_quant(rows: int, cols: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """(q uint8 [rows, cols], S float32 [cols/128, roundup(rows,4)])"""
    return (torch.empty(rows, cols, dtype=_U8, device=device),
            torch.empty(*scale_shape(rows, cols), dtype=_F, device=device))
