"""GB300 (sm_103a) row-wise RMSNorm: plain, fused residual-add, and
reduce + residual-add.

Thin Python binding over the C ABI in ``include/rarn.h`` (``librarn.so``,
built in-tree by ``residual_add_rmsnorm_gb300.build``).  This module only
checks and marshals arguments -- tensors to device pointers, the current CUDA
stream -- and raises on a non-OK status.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback: if the
library is missing or fails to load, every call raises.

    y = rms_norm(x, gamma, eps)                         # x: [..., H]
    y = fused_add_rms_norm(x, residual, gamma, eps)     # residual updated in place
    y = reduce_add_rms_norm(partials, residual, gamma, eps)   # partials: [R, ..., H]

8-bit output (e4m3 / e5m2 codes with a per-tensor or per-row scale):

    rms_norm_fp8(x, gamma, eps, out, scale, fmt="e4m3", scale_mode="tensor")
    fused_add_rms_norm_fp8(x, residual, gamma, eps, out, scale, ...)
    reduce_add_rms_norm_fp8(partials, residual, gamma, eps, out, scale, ...)
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm", "rms_norm_host",
           "fused_add_rms_norm_host", "reduce_add_rms_norm_host", "RarnError", "library",
           "set_path", "get_path", "set_pdl", "get_pdl", "plan", "watchdog", "PATHS",
           "DTYPE_CODES", "rms_norm_ex", "fused_add_rms_norm_ex", "reduce_add_rms_norm_ex",
           "rms_norm_fp8", "fused_add_rms_norm_fp8", "reduce_add_rms_norm_fp8", "plan_fp8",
           "FP8_FORMATS", "SCALE_MODES", "gemm_add_rms_norm", "plan_gemm", "plan_fp8in", "plan_tp",
           "gemm_workspace_bytes", "gemm_add_rms_norm_noalloc", "reduce_add_rms_norm_fp8in",
           "TUNING", "set_tuning", "get_tuning", "reset_tuning", "tuning", "gemm_noalloc_rows",
           "launch_floor", "tp_rows", "tp_reduce_add_rms_norm", "tp_reduce_add_rms_norm_world",
           "ipc_export", "ipc_import", "ipc_close", "TP_MAX_RANKS", "TP_SIGNAL_BYTES",
           "IPC_HANDLE_BYTES"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librarn.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
OP_CODES = {"rms_norm": 0, "fused_add_rms_norm": 1, "reduce_add_rms_norm": 2}
PATHS = {"auto": 0, "rows": 1, "stream": 2, "cluster": 3}
FP8_FORMATS = {"e4m3": 0, "e5m2": 1}
SCALE_MODES = {"tensor": 0, "row": 1}
# rarn_tuning knobs (planner overrides; -1 is the planner's own choice)
TUNING = {"rows_per_thread": 0, "rows_grid": 1, "rows_pipeline": 2, "l2_rows": 3,
          "stream_packs": 4, "stream_groups": 5, "gemm_cols": 6, "gemm_slab": 7,
          "gemm_ctas_per_sm": 8, "gemm_persistent": 9, "gemm_pair": 10,
          "gemm_norm_in_epilogue": 11, "gemm_tail_split": 12, "gemm_split_k": 13,
          "fp8in_ring": 14, "fp8in_pack16": 15, "tp_prefetch": 16}
STATUS = {0: "RARN_OK", 1: "RARN_ERR_INVALID_ARG", 2: "RARN_ERR_UNSUPPORTED",
          3: "RARN_ERR_ALIAS", 4: "RARN_ERR_CUDA"}


class RarnError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {STATUS.get(status, status)}"
        if status == 4:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


class Rows(ctypes.Structure):
    """``rarn_rows``: data pointer, row stride in elements, storage type."""
    _fields_ = [("data", ctypes.c_void_p), ("row_stride", ctypes.c_int64),
                ("dtype", ctypes.c_int)]


TP_MAX_RANKS = 8
TP_SIGNAL_BYTES = 1024 * TP_MAX_RANKS * 4
IPC_HANDLE_BYTES = 96


class TpGroup(ctypes.Structure):
    """``rarn_tp_group``: world size, rank, every rank's buffer and signal pad
    as this process addresses them."""
    _fields_ = [("world_size", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("buffers", ctypes.c_void_p * TP_MAX_RANKS),
                ("signals", ctypes.c_void_p * TP_MAX_RANKS)]


class Fp8Rows(ctypes.Structure):
    """``rarn_fp8_rows``: code matrix (row stride in bytes), format, scale
    mode and the scale's device pointer."""
    _fields_ = [("data", ctypes.c_void_p), ("row_stride", ctypes.c_int64),
                ("format", ctypes.c_int), ("scale_mode", ctypes.c_int),
                ("scale", ctypes.c_void_p)]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded ``librarn.so`` with its argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m residual_add_rmsnorm_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                ctypes.c_float, ctypes.c_int)
    lib.rarn_rms_norm.argtypes = [vp, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_fused_add_rms_norm.argtypes = [vp, vp, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_reduce_add_rms_norm.argtypes = [vp, vp, i32, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_rms_norm_host.argtypes = [vp, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_fused_add_rms_norm_host.argtypes = [vp, vp, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_reduce_add_rms_norm_host.argtypes = [vp, vp, i32, vp, vp, i64, i64, f32, c_int, vp]
    for f in (lib.rarn_rms_norm, lib.rarn_fused_add_rms_norm, lib.rarn_reduce_add_rms_norm,
              lib.rarn_rms_norm_host, lib.rarn_fused_add_rms_norm_host,
              lib.rarn_reduce_add_rms_norm_host):
        f.restype = c_int
    lib.rarn_status_string.argtypes = [c_int]
    lib.rarn_status_string.restype = ctypes.c_char_p
    lib.rarn_last_cuda_error.argtypes = []
    lib.rarn_last_cuda_error.restype = c_int
    lib.rarn_set_path.argtypes = [c_int]
    lib.rarn_set_path.restype = c_int
    lib.rarn_get_path.argtypes = []
    lib.rarn_get_path.restype = c_int
    lib.rarn_plan.argtypes = [c_int, i64, i64, i32, c_int, c_int, c_int, ctypes.c_char_p,
                              ctypes.c_size_t]
    lib.rarn_plan.restype = c_int
    lib.rarn_watchdog.argtypes = [ctypes.POINTER(ctypes.c_uint32), c_int]
    lib.rarn_watchdog.restype = c_int
    lib.rarn_version.argtypes = []
    lib.rarn_version.restype = c_int
    lib.rarn_host_access.argtypes = []
    lib.rarn_host_access.restype = c_int
    lib.rarn_rms_norm_ex.argtypes = [Rows, Rows, vp, i64, i64, f32, vp]
    lib.rarn_fused_add_rms_norm_ex.argtypes = [Rows, Rows, Rows, vp, i64, i64, f32, vp]
    lib.rarn_reduce_add_rms_norm_ex.argtypes = [Rows, Rows, i64, i32, Rows, vp, i64, i64, f32,
                                                vp]
    for f in (lib.rarn_rms_norm_ex, lib.rarn_fused_add_rms_norm_ex,
              lib.rarn_reduce_add_rms_norm_ex):
        f.restype = c_int
    lib.rarn_plan_ex.argtypes = [c_int, i64, i64, i32, c_int, c_int, c_int, c_int,
                                 ctypes.c_char_p, ctypes.c_size_t]
    lib.rarn_plan_ex.restype = c_int
    fp = ctypes.POINTER(Fp8Rows)
    lib.rarn_rms_norm_fp8.argtypes = [fp, Rows, vp, i64, i64, f32, vp]
    lib.rarn_fused_add_rms_norm_fp8.argtypes = [fp, Rows, Rows, vp, i64, i64, f32, vp]
    lib.rarn_reduce_add_rms_norm_fp8.argtypes = [fp, Rows, i64, i32, Rows, vp, i64, i64, f32, vp]
    for f in (lib.rarn_rms_norm_fp8, lib.rarn_fused_add_rms_norm_fp8,
              lib.rarn_reduce_add_rms_norm_fp8):
        f.restype = c_int
    lib.rarn_plan_fp8.argtypes = [c_int, i64, i64, i32, c_int, c_int, c_int, ctypes.c_char_p,
                                  ctypes.c_size_t]
    lib.rarn_plan_fp8.restype = c_int
    lib.rarn_gemm_add_rms_norm.argtypes = [Rows, Rows, Rows, Rows, vp, i64, i64, i64, f32, vp,
                                           ctypes.c_size_t, vp]
    lib.rarn_gemm_add_rms_norm.restype = c_int
    lib.rarn_gemm_add_rms_norm_noalloc.argtypes = [Rows, Rows, Rows, Rows, vp, i64, i64, i64,
                                                   f32, vp]
    lib.rarn_gemm_add_rms_norm_noalloc.restype = c_int
    lib.rarn_reduce_add_rms_norm_fp8in.argtypes = [vp, vp, i32, c_int, vp, vp, vp, i64, i64, f32,
                                                   c_int, vp]
    lib.rarn_reduce_add_rms_norm_fp8in.restype = c_int
    lib.rarn_gemm_workspace_bytes.argtypes = [i64, i64]
    lib.rarn_gemm_workspace_bytes.restype = i64
    lib.rarn_plan_gemm.argtypes = [i64, i64, i64, c_int, ctypes.c_int32, ctypes.c_char_p,
                                   ctypes.c_size_t]
    lib.rarn_plan_gemm.restype = c_int
    lib.rarn_plan_fp8in.argtypes = [i64, i64, ctypes.c_int32, c_int, c_int, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_char_p, ctypes.c_size_t]
    lib.rarn_plan_fp8in.restype = c_int
    lib.rarn_plan_tp.argtypes = [i64, i64, ctypes.c_int32, c_int, c_int, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_char_p, ctypes.c_size_t]
    lib.rarn_plan_tp.restype = c_int
    lib.rarn_set_pdl.argtypes = [c_int]
    lib.rarn_set_pdl.restype = c_int
    lib.rarn_get_pdl.argtypes = []
    lib.rarn_get_pdl.restype = c_int
    lib.rarn_test_stall.argtypes = [ctypes.c_longlong, ctypes.c_ulonglong]
    lib.rarn_test_stall.restype = c_int
    lib.rarn_set_tuning.argtypes = [c_int, i64]
    lib.rarn_set_tuning.restype = c_int
    lib.rarn_get_tuning.argtypes = [c_int, ctypes.POINTER(i64)]
    lib.rarn_get_tuning.restype = c_int
    lib.rarn_reset_tuning.argtypes = []
    lib.rarn_reset_tuning.restype = c_int
    tg = ctypes.POINTER(TpGroup)
    lib.rarn_tp_rows.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.rarn_tp_rows.restype = c_int
    lib.rarn_tp_reduce_add_rms_norm.argtypes = [tg, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_tp_reduce_add_rms_norm.restype = c_int
    lib.rarn_tp_reduce_add_rms_norm_world.argtypes = [tg, vp, vp, i64, i64, f32, c_int, vp]
    lib.rarn_tp_reduce_add_rms_norm_world.restype = c_int
    lib.rarn_ipc_export.argtypes = [vp, vp]
    lib.rarn_ipc_export.restype = c_int
    lib.rarn_ipc_import.argtypes = [vp, ctypes.POINTER(vp)]
    lib.rarn_ipc_import.restype = c_int
    lib.rarn_ipc_close.argtypes = [vp]
    lib.rarn_ipc_close.restype = c_int
    lib.rarn_launch_floor.argtypes = [vp, i64, i32, i32, vp]
    lib.rarn_launch_floor.restype = c_int
    lib.rarn_gemm_noalloc_rows.argtypes = [i64]
    lib.rarn_gemm_noalloc_rows.restype = i64
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise RarnError(status, what, library().rarn_last_cuda_error() if status == 4 else 0)


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}: expected float32, float16 or bfloat16")
    return codes[t.dtype]


def _check_tensor(name, t, dtype, device):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def rms_norm(x, gamma, eps: float, out=None):
    """y = x * rsqrt(mean(x^2, -1) + eps) * gamma over the last dimension.

    x: [..., H] CUDA tensor (float32 / float16 / bfloat16, contiguous);
    gamma: [H].  ``out`` may be given (it may be ``x`` itself).  Runs on the
    current stream of x's device.
    """
    import torch
    H = x.shape[-1]
    _check_tensor("x", x, x.dtype, x.device)
    _check_tensor("gamma", gamma, x.dtype, x.device)
    if gamma.numel() != H:
        raise ValueError(f"gamma has {gamma.numel()} elements, expected {H}")
    y = torch.empty_like(x) if out is None else out
    _check_tensor("out", y, x.dtype, x.device)
    if y.shape != x.shape:
        raise ValueError("out must have the shape of x")
    T = x.numel() // H if H else 0
    with torch.cuda.device(x.device):
        _check(library().rarn_rms_norm(y.data_ptr(), x.data_ptr(), gamma.data_ptr(), T, H,
                                       float(eps), _dtype_code(x), _stream(x.device)),
               "rarn_rms_norm")
    return y


def fused_add_rms_norm(x, residual, gamma, eps: float, out=None):
    """residual <- x + residual (in place); returns RMSNorm(residual) * gamma.

    x, residual: [..., H]; gamma: [H]; all one dtype, contiguous, on one CUDA
    device.  ``out`` may be ``x``.
    """
    import torch
    H = x.shape[-1]
    for n, t in (("x", x), ("residual", residual), ("gamma", gamma)):
        _check_tensor(n, t, x.dtype, x.device)
    if residual.shape != x.shape:
        raise ValueError("residual must have the shape of x")
    if gamma.numel() != H:
        raise ValueError(f"gamma has {gamma.numel()} elements, expected {H}")
    y = torch.empty_like(x) if out is None else out
    _check_tensor("out", y, x.dtype, x.device)
    if y.shape != x.shape:
        raise ValueError("out must have the shape of x")
    T = x.numel() // H if H else 0
    with torch.cuda.device(x.device):
        _check(library().rarn_fused_add_rms_norm(
            y.data_ptr(), x.data_ptr(), residual.data_ptr(), gamma.data_ptr(), T, H, float(eps),
            _dtype_code(x), _stream(x.device)), "rarn_fused_add_rms_norm")
    return y


def reduce_add_rms_norm(partials, residual, gamma, eps: float, out=None):
    """residual <- ((p_0 + p_1) + ... + p_{R-1}) + residual (binary32, one
    rounding, in place); returns RMSNorm(residual) * gamma.

    partials: [R, ..., H]; residual: [..., H]; gamma: [H].  ``out`` may be
    ``partials[0]``.
    """
    import torch
    R = partials.shape[0]
    H = residual.shape[-1]
    for n, t in (("partials", partials), ("residual", residual), ("gamma", gamma)):
        _check_tensor(n, t, residual.dtype, residual.device)
    if tuple(partials.shape[1:]) != tuple(residual.shape):
        raise ValueError("partials must have shape [R, *residual.shape]")
    if gamma.numel() != H:
        raise ValueError(f"gamma has {gamma.numel()} elements, expected {H}")
    y = torch.empty_like(residual) if out is None else out
    _check_tensor("out", y, residual.dtype, residual.device)
    if y.shape != residual.shape:
        raise ValueError("out must have the shape of residual")
    T = residual.numel() // H if H else 0
    with torch.cuda.device(residual.device):
        _check(library().rarn_reduce_add_rms_norm(
            y.data_ptr(), partials.data_ptr(), R, residual.data_ptr(), gamma.data_ptr(), T, H,
            float(eps), _dtype_code(residual), _stream(residual.device)),
            "rarn_reduce_add_rms_norm")
    return y


def _check_host(name, t, dtype):
    if t.is_cuda:
        raise ValueError(f"{name} must be a pinned host tensor")
    if not t.is_pinned():
        raise ValueError(f"{name} must be pinned (torch.Tensor.pin_memory())")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _host_call(fn, what, device):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(fn(_stream(dev)), what)


def rms_norm_host(x, gamma, eps: float, out=None, device=None):
    """rms_norm on pinned host tensors: the kernel on ``device`` (default:
    the current one) reads x and gamma and writes y through their device
    mapping; y is in host memory once that device's current stream reaches
    the call."""
    import torch
    H = x.shape[-1]
    for n, t in (("x", x), ("gamma", gamma)):
        _check_host(n, t, x.dtype)
    y = torch.empty_like(x).pin_memory() if out is None else out
    _check_host("out", y, x.dtype)
    if y.shape != x.shape or gamma.numel() != H:
        raise ValueError("shape mismatch")
    T = x.numel() // H if H else 0
    _host_call(lambda st: library().rarn_rms_norm_host(
        y.data_ptr(), x.data_ptr(), gamma.data_ptr(), T, H, float(eps), _dtype_code(x), st),
        "rarn_rms_norm_host", device)
    return y


def fused_add_rms_norm_host(x, residual, gamma, eps: float, out=None, device=None):
    """fused_add_rms_norm on pinned host tensors (see rms_norm_host)."""
    import torch
    H = x.shape[-1]
    for n, t in (("x", x), ("residual", residual), ("gamma", gamma)):
        _check_host(n, t, x.dtype)
    y = torch.empty_like(x).pin_memory() if out is None else out
    _check_host("out", y, x.dtype)
    if y.shape != x.shape or residual.shape != x.shape or gamma.numel() != H:
        raise ValueError("shape mismatch")
    T = x.numel() // H if H else 0
    _host_call(lambda st: library().rarn_fused_add_rms_norm_host(
        y.data_ptr(), x.data_ptr(), residual.data_ptr(), gamma.data_ptr(), T, H, float(eps),
        _dtype_code(x), st), "rarn_fused_add_rms_norm_host", device)
    return y


def reduce_add_rms_norm_host(partials, residual, gamma, eps: float, out=None, device=None):
    """reduce_add_rms_norm on pinned host tensors (see rms_norm_host)."""
    import torch
    R = partials.shape[0]
    H = residual.shape[-1]
    for n, t in (("partials", partials), ("residual", residual), ("gamma", gamma)):
        _check_host(n, t, residual.dtype)
    y = torch.empty_like(residual).pin_memory() if out is None else out
    _check_host("out", y, residual.dtype)
    if tuple(partials.shape[1:]) != tuple(residual.shape) or y.shape != residual.shape or \
            gamma.numel() != H:
        raise ValueError("shape mismatch")
    T = residual.numel() // H if H else 0
    _host_call(lambda st: library().rarn_reduce_add_rms_norm_host(
        y.data_ptr(), partials.data_ptr(), R, residual.data_ptr(), gamma.data_ptr(), T, H,
        float(eps), _dtype_code(residual), st), "rarn_reduce_add_rms_norm_host", device)
    return y


def set_path(name: str) -> None:
    """Force a kernel family ('auto', 'rows', 'stream', 'cluster'), process-wide."""
    _check(library().rarn_set_path(PATHS[name]), "rarn_set_path")


def _rows(name, t, device):
    """A 2-D CUDA tensor with unit element stride as a rarn_rows."""
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dim() != 2 or t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must be 2-D with unit stride along rows and a row stride "
                         f">= its row length")
    return Rows(t.data_ptr(), t.stride(0), _dtype_code(t))


def rms_norm_ex(x, gamma, eps: float, out):
    """rms_norm on row-strided 2-D views: x [T, H] and out [T, H] may be
    slices of wider tensors (unit stride within a row, any row stride >= H)."""
    import torch
    T, H = x.shape
    _check_tensor("gamma", gamma, x.dtype, x.device)
    if gamma.numel() != H or tuple(out.shape) != (T, H):
        raise ValueError("shape mismatch")
    with torch.cuda.device(x.device):
        _check(library().rarn_rms_norm_ex(_rows("out", out, x.device), _rows("x", x, x.device),
                                          gamma.data_ptr(), T, H, float(eps), _stream(x.device)),
               "rarn_rms_norm_ex")
    return out


def fused_add_rms_norm_ex(x, residual, gamma, eps: float, out):
    """fused_add_rms_norm on row-strided 2-D views; the residual may be
    float32 with float16 / bfloat16 x, gamma and out (an fp32 residual
    stream: the sum is kept in binary32)."""
    import torch
    T, H = x.shape
    _check_tensor("gamma", gamma, x.dtype, x.device)
    if gamma.numel() != H or tuple(out.shape) != (T, H) or tuple(residual.shape) != (T, H):
        raise ValueError("shape mismatch")
    with torch.cuda.device(x.device):
        _check(library().rarn_fused_add_rms_norm_ex(
            _rows("out", out, x.device), _rows("x", x, x.device),
            _rows("residual", residual, x.device), gamma.data_ptr(), T, H, float(eps),
            _stream(x.device)), "rarn_fused_add_rms_norm_ex")
    return out


def reduce_add_rms_norm_ex(partials, residual, gamma, eps: float, out):
    """reduce_add_rms_norm on strided views: partials [R, T, H] with unit
    stride within a row and any row / partial strides; residual and out are
    row-strided 2-D views; the residual may be float32 with 16-bit partials."""
    import torch
    R, T, H = partials.shape
    dev = partials.device
    if not partials.is_cuda or partials.stride(2) != 1 or partials.stride(1) < H:
        raise ValueError("partials must be [R, T, H] with unit stride within a row")
    _check_tensor("gamma", gamma, partials.dtype, dev)
    if gamma.numel() != H or tuple(out.shape) != (T, H) or tuple(residual.shape) != (T, H):
        raise ValueError("shape mismatch")
    pr = Rows(partials.data_ptr(), partials.stride(1), _dtype_code(partials))
    with torch.cuda.device(dev):
        _check(library().rarn_reduce_add_rms_norm_ex(
            _rows("out", out, dev), pr, partials.stride(0), R, _rows("residual", residual, dev),
            gamma.data_ptr(), T, H, float(eps), _stream(dev)), "rarn_reduce_add_rms_norm_ex")
    return out


def _fp8_out(out, scale, fmt, scale_mode, T, H, device):
    """The rarn_fp8_rows of an 8-bit output: ``out`` is a 2-D [T, H] view
    (unit stride within a row) of uint8 or a torch float8 type (whose format
    must then match ``fmt``); ``scale`` a float32 CUDA tensor of 1 (per
    tensor) or T (per row, contiguous) values."""
    import torch
    f8 = {torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}
    if out.dtype in f8:
        if f8[out.dtype] != fmt:
            raise ValueError(f"out is {out.dtype} but fmt is {fmt}")
    elif out.dtype != torch.uint8:
        raise TypeError("out must be uint8 or a float8 tensor")
    if not out.is_cuda or out.device != device:
        raise ValueError(f"out must be a CUDA tensor on {device}")
    if tuple(out.shape) != (T, H) or out.stride(1) != 1 or (T > 1 and out.stride(0) < H):
        raise ValueError("out must be [T, H] with unit stride within a row")
    n = 1 if scale_mode == "tensor" else T
    if (not scale.is_cuda or scale.device != device or scale.dtype != torch.float32 or
            scale.numel() != n or (n > 1 and scale.stride(0) != 1)):
        raise ValueError(f"scale must be a contiguous float32 CUDA tensor of {n} values")
    return Fp8Rows(out.data_ptr(), out.stride(0) if T > 1 else H, FP8_FORMATS[fmt],
                   SCALE_MODES[scale_mode], scale.data_ptr())


def rms_norm_fp8(x, gamma, eps: float, out, scale, fmt: str = "e4m3",
                 scale_mode: str = "tensor"):
    """RMSNorm with an 8-bit output: out[t, i] = code of v / s, v = x_i /
    RMS(x) * gamma_i, s = scale[0] (per tensor) or max|v| / maxf written to
    scale[t] (per row).  x: 2-D row-strided view."""
    import torch
    T, H = x.shape
    _check_tensor("gamma", gamma, x.dtype, x.device)
    if gamma.numel() != H:
        raise ValueError("shape mismatch")
    d = _fp8_out(out, scale, fmt, scale_mode, T, H, x.device)
    with torch.cuda.device(x.device):
        _check(library().rarn_rms_norm_fp8(ctypes.byref(d), _rows("x", x, x.device),
                                           gamma.data_ptr(), T, H, float(eps),
                                           _stream(x.device)), "rarn_rms_norm_fp8")
    return out


def fused_add_rms_norm_fp8(x, residual, gamma, eps: float, out, scale, fmt: str = "e4m3",
                           scale_mode: str = "tensor"):
    """fused_add_rms_norm with an 8-bit output (residual updated in place, of
    x's type)."""
    import torch
    T, H = x.shape
    _check_tensor("gamma", gamma, x.dtype, x.device)
    if gamma.numel() != H or tuple(residual.shape) != (T, H):
        raise ValueError("shape mismatch")
    d = _fp8_out(out, scale, fmt, scale_mode, T, H, x.device)
    with torch.cuda.device(x.device):
        _check(library().rarn_fused_add_rms_norm_fp8(
            ctypes.byref(d), _rows("x", x, x.device), _rows("residual", residual, x.device),
            gamma.data_ptr(), T, H, float(eps), _stream(x.device)), "rarn_fused_add_rms_norm_fp8")
    return out


def reduce_add_rms_norm_fp8(partials, residual, gamma, eps: float, out, scale,
                            fmt: str = "e4m3", scale_mode: str = "tensor"):
    """reduce_add_rms_norm with an 8-bit output: partials [R, T, H] with unit
    stride within a row (any row / partial strides)."""
    import torch
    R, T, H = partials.shape
    dev = partials.device
    if not partials.is_cuda or partials.stride(2) != 1 or partials.stride(1) < H:
        raise ValueError("partials must be [R, T, H] with unit stride within a row")
    _check_tensor("gamma", gamma, partials.dtype, dev)
    if gamma.numel() != H or tuple(residual.shape) != (T, H):
        raise ValueError("shape mismatch")
    d = _fp8_out(out, scale, fmt, scale_mode, T, H, dev)
    pr = Rows(partials.data_ptr(), partials.stride(1), _dtype_code(partials))
    with torch.cuda.device(dev):
        _check(library().rarn_reduce_add_rms_norm_fp8(
            ctypes.byref(d), pr, partials.stride(0), R, _rows("residual", residual, dev),
            gamma.data_ptr(), T, H, float(eps), _stream(dev)), "rarn_reduce_add_rms_norm_fp8")
    return out


def plan_fp8(op: str, T: int, H: int, R: int, dtype: str, vec_ok: bool = True,
             num_sms: int = 0) -> str:
    """The kernel the current path setting would launch for an 8-bit output."""
    buf = ctypes.create_string_buffer(256)
    st = library().rarn_plan_fp8(OP_CODES[op], T, H, R, DTYPE_CODES[dtype], int(vec_ok),
                                 num_sms, buf, 256)
    if st not in (0, 2):
        _check(st, "rarn_plan_fp8")
    return buf.value.decode()


def gemm_noalloc_rows(H: int) -> int:
    """Rows one launch sequence of gemm_add_rms_norm_noalloc covers at row
    length H (-1: H unsupported)."""
    return int(library().rarn_gemm_noalloc_rows(H))


def gemm_workspace_bytes(T: int, H: int) -> int:
    """Workspace bytes the GEMM form needs for T rows of H (-1: H unsupported)."""
    return int(library().rarn_gemm_workspace_bytes(T, H))


def gemm_add_rms_norm(a, w, residual, gamma, eps: float, out=None, workspace=None):
    """The fused form whose partial is a matrix product: P = a @ w.T
    (a [T, K], w [H, K], bfloat16 or float16; 2-D views with unit stride
    within a row), residual [T, H] <- RN(P + residual) in place,
    y = RMSNorm(residual) * gamma into ``out`` (allocated if None).
    ``workspace``: a CUDA tensor of at least gemm_workspace_bytes(T, H) bytes
    (allocated if None)."""
    import torch
    T, K = a.shape
    H = w.shape[0]
    dev = a.device
    if tuple(w.shape) != (H, K) or tuple(residual.shape) != (T, H) or gamma.numel() != H:
        raise ValueError("shape mismatch")
    _check_tensor("gamma", gamma, a.dtype, dev)
    if out is None:
        out = torch.empty(T, H, dtype=a.dtype, device=dev)
    if workspace is None:
        n = max(gemm_workspace_bytes(T, H), 4)
        workspace = torch.empty((n + 3) // 4, dtype=torch.float32, device=dev)
    if not workspace.is_cuda or workspace.device != dev:
        raise ValueError(f"workspace must be a CUDA tensor on {dev}")
    with torch.cuda.device(dev):
        _check(library().rarn_gemm_add_rms_norm(
            _rows("out", out, dev), _rows("a", a, dev), _rows("w", w, dev),
            _rows("residual", residual, dev), gamma.data_ptr(), T, H, K, float(eps),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream(dev)), "rarn_gemm_add_rms_norm")
    return out


def gemm_add_rms_norm_noalloc(a, w, residual, gamma, eps: float, out=None):
    """gemm_add_rms_norm through the entry point that allocates nothing.

    For callers that cannot allocate device memory (a plug-in whose host
    program owns all device memory, a runtime that forbids allocation once it
    serves, code that cannot take cudaMalloc's implicit synchronisation): the
    partial sums live in a 4 MiB array the library reserves on each GPU when
    it is loaded.  The first call on a device looks up that array's address;
    make it before any stream capture.  Calls on one device share the array,
    so calls that overlap on the GPU race: keep them on one stream or
    synchronise the streams.  ``out`` is allocated here only when not given;
    pass it to keep the whole call allocation-free."""
    import torch
    T, K = a.shape
    H = w.shape[0]
    dev = a.device
    if tuple(w.shape) != (H, K) or tuple(residual.shape) != (T, H) or gamma.numel() != H:
        raise ValueError("shape mismatch")
    _check_tensor("gamma", gamma, a.dtype, dev)
    if out is None:
        out = torch.empty(T, H, dtype=a.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(library().rarn_gemm_add_rms_norm_noalloc(
            _rows("out", out, dev), _rows("a", a, dev), _rows("w", w, dev),
            _rows("residual", residual, dev), gamma.data_ptr(), T, H, K, float(eps),
            _stream(dev)), "rarn_gemm_add_rms_norm_noalloc")
    return out


def reduce_add_rms_norm_fp8in(codes, scales, residual, gamma, eps: float, fmt: str = "e4m3",
                              out=None):
    """reduce_add_rms_norm over R partials stored as 8-bit codes: ``codes``
    [R, ...rows..., H] (uint8, or a torch float8 tensor of the format),
    ``scales`` [R] binary32 on the same device (partial r is code * scales[r]),
    ``residual`` [...rows..., H] updated in place; returns y like the
    residual."""
    import torch
    if codes.dtype in (getattr(torch, "float8_e4m3fn", None), getattr(torch, "float8_e5m2", None)):
        codes = codes.view(torch.uint8)
    if codes.dtype != torch.uint8:
        raise TypeError("codes must be uint8 or float8")
    R, H = codes.shape[0], residual.shape[-1]
    dev = residual.device
    if tuple(codes.shape[1:]) != tuple(residual.shape) or gamma.numel() != H:
        raise ValueError("shape mismatch")
    if scales.dtype != torch.float32 or scales.numel() != R or scales.device != dev:
        raise ValueError("scales must be R binary32 values on the residual's device")
    for n, t in (("codes", codes), ("residual", residual), ("scales", scales)):
        if t.device != dev or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous tensor on {dev}")
    _check_tensor("gamma", gamma, residual.dtype, dev)
    if out is None:
        out = torch.empty_like(residual)
    T = residual.numel() // H if H else 0
    with torch.cuda.device(dev):
        _check(library().rarn_reduce_add_rms_norm_fp8in(
            out.data_ptr(), codes.data_ptr(), R, FP8_FORMATS[fmt], scales.data_ptr(),
            residual.data_ptr(), gamma.data_ptr(), T, H, float(eps), _dtype_code(residual),
            _stream(dev)), "rarn_reduce_add_rms_norm_fp8in")
    return out


def plan_fp8in(T: int, H: int, R: int, dtype: str = "bf16", codes_aligned16: bool = True,
               num_sms: int = 152, max_smem: int = 232448) -> str:
    """The kernel reduce_add_rms_norm_fp8in takes for a problem on a device
    with `num_sms` SMs and `max_smem` bytes of opt-in shared memory per CTA
    (host logic only; the defaults are a GB300's)."""
    buf = ctypes.create_string_buffer(256)
    st = library().rarn_plan_fp8in(T, H, R, DTYPE_CODES[dtype], int(codes_aligned16), num_sms,
                                   max_smem, buf, 256)
    if st not in (0, 2):
        _check(st, "rarn_plan_fp8in")
    return buf.value.decode()


def plan_tp(T: int, H: int, N: int, dtype: str = "bf16", world: bool = True, num_sms: int = 152,
            blocks_per_sm: int = 0) -> str:
    """The launch a tensor-parallel call over N ranks makes (``world``: every
    rank's part in one launch) on a device with ``num_sms`` SMs that holds
    ``blocks_per_sm`` CTAs of the kernel per SM; 0 for either queries the
    current device (host logic only when both are given)."""
    buf = ctypes.create_string_buffer(256)
    st = library().rarn_plan_tp(T, H, N, DTYPE_CODES[dtype], int(world), num_sms, blocks_per_sm,
                                buf, 256)
    if st not in (0, 2):
        _check(st, "rarn_plan_tp")
    return buf.value.decode()


def plan_gemm(T: int, H: int, K: int, dtype: str = "bf16", num_sms: int = 152) -> str:
    """The GEMM kernel's tiling for a problem on a device with ``num_sms`` SMs
    (host logic only; the default is a GB300's; 0 queries the current
    device)."""
    buf = ctypes.create_string_buffer(256)
    st = library().rarn_plan_gemm(T, H, K, DTYPE_CODES[dtype], num_sms, buf, 256)
    if st not in (0, 2):
        _check(st, "rarn_plan_gemm")
    return buf.value.decode()


def launch_floor(grid: int, block: int, rows=None, row_bytes: int = 0) -> None:
    """The row kernels' launch floor on the current stream of ``rows``'s
    device (else the current device): ``grid`` CTAs of ``block`` threads that
    only prefetch one row each (``row_bytes`` bytes of ``rows`` per CTA),
    wait for the previous kernel and let the next launch.  A measurement aid."""
    import torch
    dev = rows.device if rows is not None else torch.device("cuda", torch.cuda.current_device())
    if rows is not None and rows.numel() * rows.element_size() < grid * row_bytes:
        raise ValueError("rows must hold grid * row_bytes bytes")
    with torch.cuda.device(dev):
        _check(library().rarn_launch_floor(rows.data_ptr() if rows is not None else None,
                                           row_bytes, grid, block, _stream(dev)),
               "rarn_launch_floor")


def _addr(x) -> int:
    """A device address: a tensor's data pointer, or an int as given."""
    return x.data_ptr() if hasattr(x, "data_ptr") else int(x)


def tp_rows(T: int, world_size: int, rank: int):
    """Rows [r0, r1) that ``rank`` of ``world_size`` owns in the tensor-parallel
    form."""
    r0, r1 = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(library().rarn_tp_rows(T, world_size, rank, ctypes.byref(r0), ctypes.byref(r1)),
           "rarn_tp_rows")
    return r0.value, r1.value


def _tp_group(buffers, rank, signals):
    g = TpGroup()
    g.world_size = len(buffers)
    g.rank = rank
    if len(buffers) > TP_MAX_RANKS:
        raise ValueError(f"at most {TP_MAX_RANKS} ranks")
    for q, b in enumerate(buffers):
        g.buffers[q] = _addr(b)
    if signals is not None:
        if len(signals) != len(buffers):
            raise ValueError("one signal pad per rank")
        for q, sg in enumerate(signals):
            g.signals[q] = _addr(sg)
    return g


def tp_reduce_add_rms_norm(buffers, rank: int, residual, gamma, eps: float, T: int,
                           signals=None):
    """This rank's part of the tensor-parallel form: ``buffers`` lists every
    rank's [T, H] buffer (tensors or device addresses as this process sees
    them; partial in, y for all T rows out), ``residual`` this rank's rows
    [r1 - r0, H] (updated in place), ``gamma`` [H]; ``signals`` every rank's
    pad (TP_SIGNAL_BYTES each) for the in-kernel barrier between ranks, or
    None when the caller orders the ranks.  Runs on the current stream of
    residual's device."""
    import torch
    H = gamma.numel()
    dev = residual.device
    _check_tensor("gamma", gamma, residual.dtype, dev)
    r0, r1 = tp_rows(T, len(buffers), rank)
    if tuple(residual.shape) != (r1 - r0, H) or not residual.is_contiguous():
        raise ValueError(f"residual must be this rank's rows, [{r1 - r0}, {H}], contiguous")
    g = _tp_group(buffers, rank, signals)
    with torch.cuda.device(dev):
        _check(library().rarn_tp_reduce_add_rms_norm(
            ctypes.byref(g), residual.data_ptr(), gamma.data_ptr(), T, H, float(eps),
            _dtype_code(residual), _stream(dev)), "rarn_tp_reduce_add_rms_norm")


def tp_reduce_add_rms_norm_world(buffers, residuals, gamma, eps: float, T: int, signals=None):
    """Every rank's part in one launch on this device (all buffers, residual
    rows and pads on it): ``residuals[q]`` is rank q's rows of the residual."""
    import torch
    H = gamma.numel()
    N = len(buffers)
    dev = gamma.device
    if len(residuals) != N:
        raise ValueError("one residual block per rank")
    for q, r in enumerate(residuals):
        r0, r1 = tp_rows(T, N, q)
        _check_tensor(f"residuals[{q}]", r, gamma.dtype, dev)
        if tuple(r.shape) != (r1 - r0, H):
            raise ValueError(f"residuals[{q}] must be [{r1 - r0}, {H}]")
    g = _tp_group(buffers, 0, signals)
    rp = (ctypes.c_void_p * N)(*[r.data_ptr() for r in residuals])
    with torch.cuda.device(dev):
        _check(library().rarn_tp_reduce_add_rms_norm_world(
            ctypes.byref(g), ctypes.cast(rp, ctypes.c_void_p), gamma.data_ptr(), T, H,
            float(eps), _dtype_code(gamma), _stream(dev)), "rarn_tp_reduce_add_rms_norm_world")


def ipc_export(x) -> bytes:
    """A handle (IPC_HANDLE_BYTES bytes) through which another process can
    address the device memory at ``x`` (a tensor or a device address)."""
    buf = ctypes.create_string_buffer(IPC_HANDLE_BYTES)
    _check(library().rarn_ipc_export(_addr(x), buf), "rarn_ipc_export")
    return buf.raw


def ipc_import(handle: bytes) -> int:
    """The address at which this process reaches the memory another process
    exported as ``handle``."""
    if len(handle) != IPC_HANDLE_BYTES:
        raise ValueError(f"an IPC handle has {IPC_HANDLE_BYTES} bytes")
    p = ctypes.c_void_p(0)
    _check(library().rarn_ipc_import(handle, ctypes.byref(p)), "rarn_ipc_import")
    return int(p.value)


def ipc_close(ptr: int) -> None:
    """Release a mapping ipc_import opened."""
    _check(library().rarn_ipc_close(ptr), "rarn_ipc_close")


def set_tuning(name: str, value: int) -> None:
    """Set one planner override (``TUNING`` names it; -1 restores the
    planner's choice).  Raises RarnError for a value outside the knob's list."""
    _check(library().rarn_set_tuning(TUNING[name], int(value)), f"rarn_set_tuning({name})")


def get_tuning(name: str) -> int:
    v = ctypes.c_int64(0)
    _check(library().rarn_get_tuning(TUNING[name], ctypes.byref(v)), "rarn_get_tuning")
    return v.value


def reset_tuning() -> None:
    """Every planner override back to the planner's choice."""
    _check(library().rarn_reset_tuning(), "rarn_reset_tuning")


class tuning:
    """Context manager: ``with tuning(gemm_pair=0): ...`` sets the named
    knobs and restores their previous values on exit."""

    def __init__(self, **knobs):
        self.knobs = knobs
        self.saved = {}

    def __enter__(self):
        for k, v in self.knobs.items():
            self.saved[k] = get_tuning(k)
            set_tuning(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            set_tuning(k, v)
        return False


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch for every later launch (process-wide)."""
    _check(library().rarn_set_pdl(int(bool(enable))), "rarn_set_pdl")


def get_pdl() -> bool:
    return bool(library().rarn_get_pdl())


def get_path() -> str:
    code = library().rarn_get_path()
    return {v: k for k, v in PATHS.items()}[code]


def plan(op: str, T: int, H: int, R: int, dtype: str, vec_ok: bool = True,
         num_sms: int = 0, rdtype: str | None = None) -> str:
    """The kernel the current path setting would launch for a problem
    (``rdtype``: the residual's storage type, default ``dtype``)."""
    buf = ctypes.create_string_buffer(256)
    st = library().rarn_plan_ex(OP_CODES[op], T, H, R, DTYPE_CODES[dtype],
                                DTYPE_CODES[rdtype or dtype], int(vec_ok), num_sms, buf, 256)
    if st not in (0, 2):
        _check(st, "rarn_plan")
    return buf.value.decode()


def watchdog(clear: bool = True) -> int:
    """Read (and by default clear) the current device's watchdog word."""
    v = ctypes.c_uint32(0)
    _check(library().rarn_watchdog(ctypes.byref(v), int(clear)), "rarn_watchdog")
    return v.value
