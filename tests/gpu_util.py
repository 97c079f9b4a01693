"""Helpers for the GPU parity tests: move storage bits to and from the device,
run the library through its Python binding, compare with the oracle.

The bar (for every element):
  * updated residual: bit-exact;
  * y: fp32 within 1e-5 relative error, fp16 / bf16 within 2 units in the
    last place, NaN exactly where the oracle has NaN.
"""
from __future__ import annotations

import numpy as np

import oracle
import residual_add_rmsnorm_gb300 as rarn
from pins import lib_decode, ulp_dist

Y_REL_TOL_F32 = 1e-5
Y_ULP_TOL_16 = 2


def torch_dtype(dtype):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_device(bits: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(bits, np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
        t = t.view(torch_dtype(dtype))
    return t.to(device)


def to_host(t, dtype: str) -> np.ndarray:
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def run_oracle(w, d):
    if w.op == "rms_norm":
        return oracle.rms_norm(d["x"], d["gamma"], w.eps, w.dtype)
    if w.op == "fused_add_rms_norm":
        return oracle.fused_add_rms_norm(d["x"], d["residual"], d["gamma"], w.eps, w.dtype)
    return oracle.reduce_add_rms_norm(d["partials"], d["residual"], d["gamma"], w.eps, w.dtype)


def run_gpu(w, d, out_is_input=False):
    """Run one problem through the binding; returns (y_bits, residual_bits)."""
    import torch
    dt = w.dtype
    g = to_device(d["gamma"], dt)
    if w.op == "rms_norm":
        x = to_device(d["x"], dt)
        y = rarn.rms_norm(x, g, w.eps, out=x if out_is_input else None)
        torch.cuda.synchronize()
        return to_host(y, dt), None
    res = to_device(d["residual"], dt)
    if w.op == "fused_add_rms_norm":
        x = to_device(d["x"], dt)
        y = rarn.fused_add_rms_norm(x, res, g, w.eps, out=x if out_is_input else None)
    else:
        p = to_device(d["partials"], dt)
        y = rarn.reduce_add_rms_norm(p, res, g, w.eps, out=p[0] if out_is_input else None)
    torch.cuda.synchronize()
    return to_host(y, dt), to_host(res, dt)


def assert_y_close(got: np.ndarray, want: np.ndarray, dtype: str, what=""):
    if got.size == 0:
        return
    if dtype == "f32":
        g = got.astype(np.float64)
        o = want.astype(np.float64)
        nan_o = np.isnan(o)
        assert np.array_equal(np.isnan(g), nan_o), f"{what}: NaN pattern differs"
        g, o = g[~nan_o], o[~nan_o]
        rel = np.abs(g - o) / np.maximum(np.abs(o), np.finfo(np.float32).tiny)
        worst = float(rel.max()) if rel.size else 0.0
        assert worst <= Y_REL_TOL_F32, f"{what}: max rel err {worst:.3e}"
    else:
        # NaN exactly where the oracle has NaN (payloads are not specified);
        # the other elements within 2 ulps
        nan_o = np.isnan(lib_decode(want, dtype))
        assert np.array_equal(np.isnan(lib_decode(got, dtype)), nan_o), \
            f"{what}: NaN pattern differs"
        d = ulp_dist(np.asarray(got)[~nan_o], np.asarray(want)[~nan_o], dtype)
        worst = int(d.max()) if d.size else 0
        assert worst <= Y_ULP_TOL_16, f"{what}: max ulp distance {worst}"


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    g = np.ascontiguousarray(got).view(np.uint8)
    w = np.ascontiguousarray(want).view(np.uint8)
    if not np.array_equal(g, w):
        n = np.count_nonzero(np.ascontiguousarray(got).ravel().view(np.uint16 if got.itemsize == 2
                                                                     else np.uint32)
                             != np.ascontiguousarray(want).ravel().view(
                                 np.uint16 if want.itemsize == 2 else np.uint32))
        raise AssertionError(f"{what}: {n} elements differ")


def check_parity(w, d, *, out_is_input=False, what=""):
    ref = run_oracle(w, d)
    y, res = run_gpu(w, d, out_is_input=out_is_input)
    assert_y_close(y, ref.y, w.dtype, what or w.name)
    if ref.residual is not None:
        assert_bits_equal(res, ref.residual, (what or w.name) + " residual")
    return y, res


# 8-bit codes: the kernel computes v in binary32, the oracle in binary64, so
# a code may differ only where the oracle's exact u = v / s lies within
# Q_MID_REL of the midpoint between two adjacent codes' values, and then by
# one step.  (Binary32 error of v: the sum of squares over <= 2^17 terms with
# per-thread runs of <= 64 and a <= 10-level tree, rsqrtf, two products and
# the scale multiply: well below 8e-6 relative.)
Q_MID_REL = 8e-6
Q_SCALE_REL = 4e-6


def assert_codes_close(got: np.ndarray, want: np.ndarray, u64: np.ndarray, fmt: str, what=""):
    got = np.asarray(got, np.uint8)
    want = np.asarray(want, np.uint8)
    diff = got != want
    if not diff.any():
        return
    g = got[diff].astype(np.int64)
    w = want[diff].astype(np.int64)
    gv = oracle.default().decode_fp8(got[diff], fmt)
    wv = oracle.default().decode_fp8(want[diff], fmt)
    adjacent = ((g & 0x80) == (w & 0x80)) & (np.abs((g & 0x7F) - (w & 0x7F)) == 1)
    mid = (gv + wv) / 2
    near = np.abs(u64[diff] - mid) <= Q_MID_REL * np.abs(mid)
    bad = ~(adjacent & near)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} codes differ beyond a "
                           f"midpoint tie, e.g. got {g[bad][:4]} want {w[bad][:4]} "
                           f"u {u64[diff][bad][:4]}")


def assert_scales_close(got: np.ndarray, want: np.ndarray, what=""):
    rel = np.abs(got.astype(np.float64) - want) / np.abs(want.astype(np.float64))
    assert float(rel.max(initial=0.0)) <= Q_SCALE_REL, f"{what}: scale rel err {rel.max():.3e}"
