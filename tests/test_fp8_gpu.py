"""GPU parity of the 8-bit output forms (e4m3 / e5m2 codes with a per-tensor
or per-row scale) against the CPU oracle, through the Python binding and the
C ABI.

Bar: the residual bit-exact; every code equal to the oracle's, or the
adjacent code where the oracle's exact value lies within a few binary32
roundings of the midpoint between the two; per-row scales within 4e-6
relative; every byte outside the written rows untouched."""
import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import (assert_bits_equal, assert_codes_close, assert_scales_close, to_device,
                      to_host)

pytestmark = pytest.mark.gpu

FILL = {"f32": np.float32(-7.0), "f16": np.uint16(0xC700), "bf16": np.uint16(0xC0E0)}
QFILL = 0x5A
SCALES = {"e4m3": 0.01, "e5m2": 2.0 ** -12}  # a few elements saturate


@pytest.fixture(autouse=True)
def _reset_path():
    yield
    rarn.set_path("auto")
    rarn.set_pdl(True)


def _flat(rows, ld, dt, extra=0):
    """[T, H] storage into a flat buffer with row stride ld, padding = FILL."""
    T, H = rows.shape
    buf = np.full(T * ld + extra, FILL[dt], dtype=rows.dtype)
    buf[:T * ld].reshape(T, ld)[:, :H] = rows
    return buf


def run_fp8(w, d, fmt, mode, ldx=None, ldr=None, ldq=None, pextra=0, scale=None, out8=False):
    """One problem through the binding and the oracle on the same flat
    buffers; checks everything and returns the plan text."""
    import torch
    dt, T, H = w.dtype, w.T, w.H
    R = {"rms_norm": 0, "fused_add_rms_norm": 1}.get(w.op, w.R)
    ldx, ldr, ldq = ldx or H, ldr or H, ldq or H
    scale = float(np.float32(SCALES[fmt] if scale is None else scale))
    parts = d["partials"] if R > 1 else d["x"][None]
    n = max(R, 1)
    slice_ = T * ldx + pextra
    X = np.concatenate([_flat(parts[r], ldx, dt, extra=pextra) for r in range(n)])
    Rf = _flat(d["residual"], ldr, dt, extra=3) if R else None

    ref_res = None if Rf is None else Rf.copy()  # updated in place by the oracle
    codes, rs, u = oracle.rows_fp8(dt, fmt, T, H, R, X.copy(), ldx, slice_, ref_res, ldr,
                                   d["gamma"], w.eps, mode, scale, ldq, fill=QFILL,
                                   want_u64=True)

    Xd = to_device(X, dt)
    g = to_device(d["gamma"], dt)
    qdt = torch.uint8
    if out8:
        qdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    Q = torch.full((T * ldq + 7,), QFILL, dtype=torch.uint8, device="cuda")
    q = Q[:T * ldq].view(T, ldq)[:, :H]
    if out8:
        q = q.view(qdt)
    sc = (torch.tensor([scale], dtype=torch.float32, device="cuda") if mode == "tensor"
          else torch.full((T,), -1.0, dtype=torch.float32, device="cuda"))
    x = Xd[:T * ldx].view(T, ldx)[:, :H]
    if R == 0:
        rarn.rms_norm_fp8(x, g, w.eps, q, sc, fmt, mode)
    else:
        Rd = to_device(Rf, dt)
        res = Rd[:T * ldr].view(T, ldr)[:, :H]
        if R == 1:
            rarn.fused_add_rms_norm_fp8(x, res, g, w.eps, q, sc, fmt, mode)
        else:
            pv = Xd.as_strided((R, T, H), (slice_, ldx, 1))
            rarn.reduce_add_rms_norm_fp8(pv, res, g, w.eps, q, sc, fmt, mode)
    torch.cuda.synchronize()
    what = f"{w.op} {dt} T{T} H{H} {fmt} {mode}"
    Qh = Q.cpu().numpy()
    got = Qh[:T * ldq].reshape(T, ldq)
    assert np.all(got[:, H:] == QFILL) and np.all(Qh[T * ldq:] == QFILL), what + ": padding"
    assert_codes_close(got[:, :H], codes[:, :H], u, fmt, what)
    if mode == "row":
        assert_scales_close(sc.cpu().numpy(), rs, what)
    else:
        assert float(sc.item()) == scale, what + ": per-tensor scale written"
    if R:
        assert_bits_equal(to_host(Rd, dt), ref_res, what + " residual (with padding)")
    return rarn.plan_fp8(w.op, T, H, R, dt, vec_ok=True)


SHAPES = [  # T, H -- warp, pipelined warp, pipelined / single-wave CTA, scalar, two-pass
    (7, 64), (20000, 256), (3000, 4096), (100, 5120), (5, 1591), (129, 8191), (3, 100000),
]
COMBOS = [("e4m3", "tensor"), ("e4m3", "row"), ("e5m2", "tensor"), ("e5m2", "row")]


@pytest.mark.parametrize("fmt,mode", COMBOS)
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"])
def test_fp8_parity(op, dt, fmt, mode):
    kinds = set()
    for T, H in SHAPES:
        w = W.workload(op, dt, T, H, R=3, eps=1e-6, seed=T + 3 * H)
        p = run_fp8(w, W.generate(w), fmt, mode)
        kinds.add(p.split()[0] + (" pipe" if "pipe=1" in p else ""))
    assert {"rows.warp", "rows.cta", "rows.two_pass"} <= {k.split()[0] for k in kinds}, kinds


STRIDED = [  # T, H, ldx, ldr, ldq, partial-stride extra
    (33, 512, 576, 520, 640, 64),      # warp, strided packs
    (3000, 4096, 4160, 4104, 4112, 8),  # pipelined CTA
    (17, 1000, 1003, 1001, 1005, 1),   # not 16-byte strides: scalar
    (40, 2048, 2048, 2048, 2049, 0),   # codes stride odd: scalar
]


@pytest.mark.parametrize("mode", ["tensor", "row"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"])
def test_fp8_strided(op, mode):
    for T, H, ldx, ldr, ldq, pextra in STRIDED:
        for dt in ("bf16", "f32"):
            w = W.workload(op, dt, T, H, R=2, eps=1e-5, seed=T * H)
            run_fp8(w, W.generate(w), "e4m3", mode, ldx, ldr, ldq, pextra)


def test_fp8_special_rows():
    """A row of zeros (scale 1, zero codes), a row with one dominant element,
    and rows whose values all saturate under a small per-tensor scale."""
    for dt in ("bf16", "f16", "f32"):
        for T, H in ((6, 64), (6, 4096), (6, 1000)):
            w = W.workload("fused_add_rms_norm", dt, T, H, eps=1e-6, seed=H)
            d = W.generate(w)
            zero = W.to_storage(np.zeros(H), dt)
            d["x"][0] = zero
            d["residual"][0] = zero
            d["x"][1] = W.to_storage(np.where(np.arange(H) == 5, 1e3, 0.01), dt)
            d["residual"][1] = zero
            for fmt, mode in COMBOS:
                run_fp8(w, {k: v.copy() for k, v in d.items()}, fmt, mode)
            run_fp8(w, {k: v.copy() for k, v in d.items()}, "e4m3", "tensor", scale=1e-4)


def test_fp8_float8_tensor_output():
    """A torch float8 output tensor is written with the same codes, and its
    values dequantise to within the format's rounding of the 16-bit path."""
    import torch
    for fmt in ("e4m3", "e5m2"):
        w = W.workload("rms_norm", "bf16", 300, 2048, eps=1e-6, seed=1)
        run_fp8(w, W.generate(w), fmt, "row", out8=True)
    x = torch.randn(64, 4096, device="cuda", dtype=torch.bfloat16)
    g = torch.rand(4096, device="cuda", dtype=torch.bfloat16) + 0.5
    y16 = rarn.rms_norm(x, g, 1e-6).float()
    q = torch.empty(64, 4096, dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.empty(64, dtype=torch.float32, device="cuda")
    rarn.rms_norm_fp8(x, g, 1e-6, q, s, "e4m3", "row")
    deq = q.float() * s[:, None]
    # e4m3 has 4 significant bits: half a step is 1/16 relative, plus the
    # bf16 rounding of the 16-bit path
    assert torch.all((deq - y16).abs() <= y16.abs() / 16 * 1.01 + s[:, None] * 2 ** -9)


@pytest.mark.parametrize("pdl", [True, False])
def test_fp8_chained_launches(pdl):
    """Back-to-back launches on one stream: the per-tensor scale is written by
    the kernel before (a per-row launch's output feeds the next call), the
    residual chain carries over."""
    import torch
    rarn.set_pdl(pdl)
    T, H = 2000, 4096
    x = torch.randn(T, H, device="cuda", dtype=torch.bfloat16)
    res = torch.randn(T, H, device="cuda", dtype=torch.bfloat16)
    g = torch.rand(H, device="cuda", dtype=torch.bfloat16) + 0.5
    res_ref = res.clone()
    q1 = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    q2 = torch.empty_like(q1)
    s_row = torch.empty(T, dtype=torch.float32, device="cuda")
    s_t = torch.empty(1, dtype=torch.float32, device="cuda")
    for _ in range(3):
        rarn.fused_add_rms_norm_fp8(x, res, g, 1e-6, q1, s_row, "e4m3", "row")
        torch.amax(s_row, dim=0, keepdim=True, out=s_t)
        rarn.rms_norm_fp8(res, g, 1e-6, q2, s_t, "e4m3", "tensor")
    torch.cuda.synchronize()
    # the same chain with the 16-bit fused form gives the same residual
    y16 = torch.empty_like(x)
    for _ in range(3):
        rarn.fused_add_rms_norm(x, res_ref, g, 1e-6, out=y16)
    torch.cuda.synchronize()
    assert torch.equal(res, res_ref)
    # the last per-tensor launch used the last per-row scales' maximum:
    # every code's value times that scale is within e4m3 rounding of y
    y = rarn.rms_norm(res, g, 1e-6).float()
    deq = q2.view(torch.float8_e4m3fn).float() * s_t
    assert torch.all((deq - y).abs() <= y.abs() / 16 * 1.01 + s_t * 2 ** -9 + 1e-6)


@pytest.mark.parametrize("name", [w.name for w in W.EXTENDED if w.qfmt])
def test_fp8_full_size_sampled(name):
    """The 8-bit benchmark workloads at full size in the benchmark's launch
    configuration; the oracle checks every 16th row (rows are independent)."""
    import torch
    w = W.BY_NAME[name]
    d = W.generate(w)
    T, H = w.T, w.H
    fmt, mode = w.qfmt, w.qmode
    dt = w.dtype
    x = to_device(d["x"], dt)
    res = to_device(d["residual"], dt)
    g = to_device(d["gamma"], dt)
    q = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    scale = float(np.float32(w.qscale))
    sc = (torch.tensor([scale], dtype=torch.float32, device="cuda") if mode == "tensor"
          else torch.empty(T, dtype=torch.float32, device="cuda"))
    rarn.fused_add_rms_norm_fp8(x, res, g, w.eps, q, sc, fmt, mode)
    torch.cuda.synchronize()
    rows = np.arange(0, T, 16)
    xs, rs_in = d["x"][rows].copy(), d["residual"][rows].copy()
    codes, rs, u = oracle.rows_fp8(dt, fmt, len(rows), H, 1, xs.reshape(-1), H, len(rows) * H,
                                   rs_in.reshape(-1), H, d["gamma"], w.eps, mode, scale,
                                   want_u64=True)
    got = q.cpu().numpy()[rows]
    assert_codes_close(got, codes, u, fmt, name)
    assert_bits_equal(to_host(res, dt)[rows], rs_in.reshape(len(rows), H), name + " residual")
    if mode == "row":
        assert_scales_close(sc.cpu().numpy()[rows], rs, name)
