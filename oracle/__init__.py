"""CPU oracle for row-wise RMSNorm, fused residual-add RMSNorm and
reduce + residual-add RMSNorm.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``residual_add_rmsnorm_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``rarn_oracle.c`` (plain C, binary64 except for the
binary32 partial/residual sum the method prescribes); this module only
marshals numpy arrays through ctypes.  Arrays hold the raw storage bits:
``np.float32`` for f32 and ``np.uint16`` for f16 / bf16.

Sources followed (by page title and section):
  * "RMSNorm kernel", 1 Background / 2 Abstraction: y = x * gamma / RMS(x),
    RMS over the last dimension, mean of squares plus eps under the root.
  * "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: sum the partial
    buffers, add the residual, write the sum back as the residual, take the
    squares of that stored value, rsqrt(variance / hidden_size + eps), then
    scale by the reciprocal RMS and the weight.

The tensor-parallel form (``tp_reduce_add_rms_norm``) follows the tokenweave
kernel's reduce-scatter / norm / all-gather over N ranks' buffers, with rank r
owning rows floor(rT/N) .. floor((r+1)T/N)-1 and the partials summed in rank
order.

The 8-bit output (``rows_fp8``) follows "Block All Reduce", FP8 section: e4m3
and e5m2 codes, converted with saturation to the largest finite value; the
scale is a given per-tensor value or max |v| / maxf per row.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
fixed by the formats' definitions, closed forms and exact rational arithmetic.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
FP8 = {"e4m3": 0, "e5m2": 1}
QMODES = {"tensor": 0, "row": 1}


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc < 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return rc


class Result:
    """Outputs of one oracle call.

    y         storage bits of the normalised output, shape [T, H]
    residual  storage bits of the updated residual (fused / reduce), or None
    inv       binary64 reciprocal RMS per row, shape [T]
    y64       binary64 output before its final rounding (only if requested)
    threads   host threads the call used
    """

    def __init__(self, y, residual, inv, y64, threads):
        self.y, self.residual, self.inv, self.y64, self.threads = y, residual, inv, y64, threads


class Oracle:
    """ctypes front end of one build of ``rarn_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        p, i64, i32, f32, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                   ctypes.c_float, ctypes.c_int)
        lib.oracle_rms_norm.argtypes = [c_int, i64, i64, p, p, f32, p, p, p, c_int]
        lib.oracle_fused_add_rms_norm.argtypes = [c_int, i64, i64, p, p, p, f32, p, p, p, p, c_int]
        lib.oracle_reduce_add_rms_norm.argtypes = [c_int, i64, i64, i32, p, p, p, f32, p, p, p, p,
                                                   c_int]
        for f in (lib.oracle_rms_norm, lib.oracle_fused_add_rms_norm,
                  lib.oracle_reduce_add_rms_norm):
            f.restype = c_int
        lib.oracle_rows_ex.argtypes = [c_int, c_int, i64, i64, i32, p, i64, i64, p, p, i64, p, f32,
                                       p, i64, p, p, c_int]
        lib.oracle_rows_ex.restype = c_int
        lib.oracle_rows_fp8.argtypes = [c_int, c_int, i64, i64, i32, p, i64, i64, p, i64, p, f32,
                                        c_int, f32, p, i64, p, p]
        lib.oracle_rows_fp8.restype = c_int
        lib.oracle_reduce_fp8in.argtypes = [c_int, c_int, i64, i64, i32, p, p, p, p, f32, p, p, p,
                                            p, c_int]
        lib.oracle_reduce_fp8in.restype = c_int
        lib.oracle_decode_fp8.argtypes = [c_int, p, p, i64]
        lib.oracle_decode_fp8.restype = c_int
        lib.oracle_round_fp8.argtypes = [c_int, p, p, i64]
        lib.oracle_round_fp8.restype = c_int
        lib.oracle_gemm_add_rms_norm.argtypes = [c_int, i64, i64, i64, p, i64, p, i64, p, i64, p,
                                                 f32, p, i64, p, p, p, c_int]
        lib.oracle_gemm_add_rms_norm.restype = c_int
        lib.oracle_tp_reduce_add_rms_norm.argtypes = [c_int, i64, i64, i32, p, p, p, f32, p, p,
                                                      p, p, c_int]
        lib.oracle_tp_reduce_add_rms_norm.restype = c_int
        lib.oracle_tp_rows.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.oracle_tp_rows.restype = None
        lib.oracle_decode.argtypes = [c_int, p, p, i64]
        lib.oracle_decode.restype = None
        lib.oracle_round.argtypes = [c_int, p, p, i64]
        lib.oracle_round.restype = None
        self.lib = lib
        self.path = lib_path

    @staticmethod
    def _as_storage(a, dtype):
        a = np.ascontiguousarray(a)
        want = STORAGE[dtype]
        if a.dtype != want:
            raise TypeError(f"oracle expects {np.dtype(want).name} storage bits for {dtype}, "
                            f"got {a.dtype}")
        return a

    def rms_norm(self, x, gamma, eps, dtype, *, want_y64=False, threads=0) -> Result:
        x = self._as_storage(x, dtype)
        gamma = self._as_storage(gamma, dtype)
        T, H = x.shape
        y = np.empty_like(x)
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        n = _check(self.lib.oracle_rms_norm(DTYPES[dtype], T, H, _ptr(x), _ptr(gamma), float(eps),
                                            _ptr(y), _ptr(inv), _ptr(y64), threads))
        return Result(y, None, inv, y64, n)

    def fused_add_rms_norm(self, x, residual, gamma, eps, dtype, *, want_y64=False,
                           threads=0) -> Result:
        x = self._as_storage(x, dtype)
        residual = self._as_storage(residual, dtype)
        gamma = self._as_storage(gamma, dtype)
        T, H = x.shape
        y = np.empty_like(x)
        res_out = np.empty_like(x)
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        n = _check(self.lib.oracle_fused_add_rms_norm(
            DTYPES[dtype], T, H, _ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(res_out),
            _ptr(y), _ptr(inv), _ptr(y64), threads))
        return Result(y, res_out, inv, y64, n)

    def reduce_add_rms_norm(self, partials, residual, gamma, eps, dtype, *, want_y64=False,
                            threads=0) -> Result:
        partials = self._as_storage(partials, dtype)
        residual = self._as_storage(residual, dtype)
        gamma = self._as_storage(gamma, dtype)
        R, T, H = partials.shape
        y = np.empty_like(residual)
        res_out = np.empty_like(residual)
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        n = _check(self.lib.oracle_reduce_add_rms_norm(
            DTYPES[dtype], T, H, R, _ptr(partials), _ptr(residual), _ptr(gamma), float(eps),
            _ptr(res_out), _ptr(y), _ptr(inv), _ptr(y64), threads))
        return Result(y, res_out, inv, y64, n)

    def rows_ex(self, dtype, rdtype, T, H, R, x, ldx, slice_, residual, ldr, gamma, eps, y, ldy,
                *, want_y64=False, threads=0) -> Result:
        """General form: x (R = 0 or 1) or the R partials live in the flat
        storage array ``x`` with row stride ``ldx`` and ``slice_`` elements
        between partials; ``residual`` (storage type ``rdtype``, row stride
        ``ldr``) is updated IN PLACE; ``y`` (row stride ``ldy``) receives the
        first H elements of each row.  R = 0 is plain RMSNorm."""
        x = self._as_storage(x, dtype)
        gamma = self._as_storage(gamma, dtype)
        if not (y.flags.c_contiguous and y.dtype == STORAGE[dtype]):
            raise TypeError("y must be contiguous storage of the x dtype")
        if residual is not None and not (residual.flags.c_contiguous and
                                         residual.dtype == STORAGE[rdtype]):
            raise TypeError("residual must be contiguous storage of its dtype")
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        n = _check(self.lib.oracle_rows_ex(
            DTYPES[dtype], DTYPES[rdtype], T, H, R, _ptr(x), ldx, slice_, _ptr(residual),
            _ptr(residual), ldr, _ptr(gamma), float(eps), _ptr(y), ldy, _ptr(inv), _ptr(y64),
            threads))
        return Result(y, residual, inv, y64, n)

    def rows_fp8(self, dtype, fmt, T, H, R, x, ldx, slice_, residual, ldr, gamma, eps, mode,
                 scale=1.0, ldq=None, *, fill=0, want_u64=False):
        """8-bit output (``fmt`` "e4m3" / "e5m2").  x (R = 0 or 1) or the R
        partials live in the flat storage array ``x`` (row stride ``ldx``,
        ``slice_`` elements between partials); ``residual`` (row stride
        ``ldr``) is updated IN PLACE.  ``mode`` "tensor" divides by the given
        ``scale``, "row" by max|v| / maxf per row.  Returns (codes [T, ldq]
        uint8 with the padding left at ``fill``, row scales [T] float32 (row
        mode), u64 [T, H] or None)."""
        x = self._as_storage(x, dtype)
        gamma = self._as_storage(gamma, dtype)
        if residual is not None and not (residual.flags.c_contiguous and
                                         residual.dtype == STORAGE[dtype]):
            raise TypeError("residual must be contiguous storage of the x dtype")
        ldq = ldq or H
        codes = np.full(T * ldq, fill, np.uint8)
        rs = np.zeros(T, np.float32)
        u64 = np.empty((T, H), np.float64) if want_u64 else None
        _check(self.lib.oracle_rows_fp8(DTYPES[dtype], FP8[fmt], T, H, R, _ptr(x), ldx, slice_,
                                        _ptr(residual), ldr, _ptr(gamma), float(eps),
                                        QMODES[mode], float(scale), _ptr(codes), ldq, _ptr(rs),
                                        _ptr(u64)))
        return codes.reshape(T, ldq), rs, u64

    def reduce_fp8in(self, codes, scales, residual, gamma, eps, dtype, fmt, *, want_y64=False,
                     threads=0) -> Result:
        """Reduce + residual + RMSNorm over R partials of 8-bit codes
        (``codes`` uint8 [R, T, H], ``fmt`` "e4m3" / "e5m2") with one binary32
        scale per partial (``scales`` [R])."""
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.float32)
        residual = self._as_storage(residual, dtype)
        gamma = self._as_storage(gamma, dtype)
        R, T, H = codes.shape
        if scales.shape != (R,) or residual.shape != (T, H):
            raise ValueError("shape mismatch")
        y = np.zeros_like(residual)
        res_out = np.zeros_like(residual)  # zeros: a row never stored shows
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        n = _check(self.lib.oracle_reduce_fp8in(
            DTYPES[dtype], FP8[fmt], T, H, R, _ptr(codes), _ptr(scales), _ptr(residual),
            _ptr(gamma), float(eps), _ptr(res_out), _ptr(y), _ptr(inv), _ptr(y64), threads))
        return Result(y, res_out, inv, y64, n)

    def decode_fp8(self, codes, fmt) -> np.ndarray:
        """8-bit codes -> binary64 values (the oracle's own decoder)."""
        codes = np.ascontiguousarray(codes, np.uint8)
        out = np.empty(codes.shape, np.float64)
        _check(self.lib.oracle_decode_fp8(FP8[fmt], _ptr(codes), _ptr(out), codes.size))
        return out

    def round_fp8(self, values, fmt) -> np.ndarray:
        """binary64 values -> 8-bit codes, nearest-even with saturation."""
        values = np.ascontiguousarray(values, np.float64)
        out = np.empty(values.shape, np.uint8)
        _check(self.lib.oracle_round_fp8(FP8[fmt], _ptr(values), _ptr(out), values.size))
        return out

    def gemm_add_rms_norm(self, dtype, A, W, residual, gamma, eps, T, H, K, lda=None, ldw=None,
                          ldr=None, ldy=None, *, want_p64=False, threads=0):
        """GEMM producer + fused residual-add RMSNorm: P = A W^T (A: T rows of
        lda, W: H rows of ldw, flat storage arrays), h = RN(P + residual),
        residual updated IN PLACE (T rows of ldr), y returned as T rows of
        ldy.  Returns a Result with y, residual, inv, and (want_p64) the
        attributes p64 (P) and abs64 (sum |A W|), both [T, H]."""
        lda, ldw, ldr, ldy = lda or K, ldw or K, ldr or H, ldy or H
        A = self._as_storage(A, dtype)
        W = self._as_storage(W, dtype)
        gamma = self._as_storage(gamma, dtype)
        if not (residual.flags.c_contiguous and residual.dtype == STORAGE[dtype]):
            raise TypeError("residual must be contiguous storage of the dtype")
        y = np.zeros(T * ldy, STORAGE[dtype])
        inv = np.empty(T, np.float64)
        p64 = np.empty((T, H), np.float64) if want_p64 else None
        a64 = np.empty((T, H), np.float64) if want_p64 else None
        n = _check(self.lib.oracle_gemm_add_rms_norm(
            DTYPES[dtype], T, H, K, _ptr(A), lda, _ptr(W), ldw, _ptr(residual), ldr, _ptr(gamma),
            float(eps), _ptr(y), ldy, _ptr(p64), _ptr(a64), _ptr(inv), threads))
        r = Result(y, residual, inv, None, n)
        r.p64, r.abs64 = p64, a64
        return r

    def tp_rows(self, T, N, r):
        """Rows [r0, r1) that rank r of N owns in the tensor-parallel form."""
        r0, r1 = ctypes.c_int64(0), ctypes.c_int64(0)
        self.lib.oracle_tp_rows(T, N, r, ctypes.byref(r0), ctypes.byref(r1))
        return r0.value, r1.value

    def tp_reduce_add_rms_norm(self, bufs, residual, gamma, eps, dtype, *, want_y64=False,
                               threads=0):
        """Tensor-parallel form over N ranks: ``bufs`` is N partials [T, H]
        (one per rank), ``residual`` [T, H] the ranks' residual rows stacked in
        rank order.  Returns a Result whose ``ys`` is the N ranks' output
        buffers after the all-gather (``y`` is rank 0's) and ``residual`` the
        updated residual."""
        bufs = [self._as_storage(b, dtype) for b in bufs]
        residual = self._as_storage(residual, dtype)
        gamma = self._as_storage(gamma, dtype)
        N = len(bufs)
        T, H = residual.shape
        if any(b.shape != (T, H) for b in bufs):
            raise ValueError("every rank's buffer must be [T, H]")
        ys = [np.zeros_like(residual) for _ in range(N)]
        res_out = np.zeros_like(residual)
        inv = np.empty(T, np.float64)
        y64 = np.empty((T, H), np.float64) if want_y64 else None
        bp = (ctypes.c_void_p * N)(*[b.ctypes.data for b in bufs])
        yp = (ctypes.c_void_p * N)(*[y.ctypes.data for y in ys])
        n = _check(self.lib.oracle_tp_reduce_add_rms_norm(
            DTYPES[dtype], T, H, N, ctypes.cast(bp, ctypes.c_void_p), _ptr(residual),
            _ptr(gamma), float(eps), _ptr(res_out), ctypes.cast(yp, ctypes.c_void_p), _ptr(inv),
            _ptr(y64), threads))
        r = Result(ys[0], res_out, inv, y64, n)
        r.ys = ys
        return r

    def decode(self, bits, dtype) -> np.ndarray:
        """Storage bits -> binary64 values (the oracle's own decoder)."""
        bits = self._as_storage(bits, dtype)
        out = np.empty(bits.shape, np.float64)
        self.lib.oracle_decode(DTYPES[dtype], _ptr(bits), _ptr(out), bits.size)
        return out

    def round_to(self, values, dtype) -> np.ndarray:
        """binary64 values -> storage bits, one round-to-nearest-even."""
        values = np.ascontiguousarray(values, np.float64)
        out = np.empty(values.shape, STORAGE[dtype])
        self.lib.oracle_round(DTYPES[dtype], _ptr(values), _ptr(out), values.size)
        return out


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def rms_norm(*a, **k) -> Result:
    return default().rms_norm(*a, **k)


def fused_add_rms_norm(*a, **k) -> Result:
    return default().fused_add_rms_norm(*a, **k)


def reduce_add_rms_norm(*a, **k) -> Result:
    return default().reduce_add_rms_norm(*a, **k)


def rows_ex(*a, **k) -> Result:
    return default().rows_ex(*a, **k)


def rows_fp8(*a, **k):
    return default().rows_fp8(*a, **k)


def reduce_fp8in(*a, **k) -> Result:
    return default().reduce_fp8in(*a, **k)


def gemm_add_rms_norm(*a, **k) -> Result:
    return default().gemm_add_rms_norm(*a, **k)


def tp_reduce_add_rms_norm(*a, **k) -> Result:
    return default().tp_reduce_add_rms_norm(*a, **k)


def tp_rows(*a, **k):
    return default().tp_rows(*a, **k)


def decode(*a, **k) -> np.ndarray:
    return default().decode(*a, **k)


def round_to(*a, **k) -> np.ndarray:
    return default().round_to(*a, **k)


def cores() -> int:
    """Host threads the oracle uses by default."""
    return os.cpu_count() or 1
