"""GPU parity of the general forms: per-buffer row strides and an fp32
residual stream with 16-bit inputs, against the CPU oracle.  Residual
bit-exact (binary32 residual: the binary32 sum itself), y within 2 ulps /
1e-5, padding between rows untouched."""
import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import assert_bits_equal, assert_y_close, run_oracle, to_device, to_host

pytestmark = pytest.mark.gpu

FILL = -7.0


@pytest.fixture(autouse=True)
def _reset_path():
    yield
    rarn.set_path("auto")


def _strided(bits, ld, dt, extra=0):
    """Device buffer with row stride ld holding `bits` [T, H]; the padding
    and `extra` trailing elements hold FILL.  Returns (buffer, [T, H] view)."""
    import torch
    T, H = bits.shape
    dense = to_device(bits, dt)
    buf = torch.full((T * ld + extra,), FILL, dtype=dense.dtype, device=dense.device)
    view = buf[:T * ld].view(T, ld)[:, :H]
    view.copy_(dense)
    return buf, view


def _padding_untouched(buf, T, H, ld):
    import torch
    rows = buf[:T * ld].view(T, ld)
    return bool(torch.all(rows[:, H:] == FILL)) and bool(torch.all(buf[T * ld:] == FILL))


def _run_strided(w, d, ldx, ldr, ldy, pextra=0):
    """Run the general entry point on strided copies; returns host bits of y
    and the residual ([T, H]) and whether all padding stayed untouched."""
    import torch
    dt, T, H = w.dtype, w.T, w.H
    g = to_device(d["gamma"], dt)
    ybuf, y = _strided(np.zeros((T, H), d["gamma"].dtype), ldy, dt, extra=5)
    untouched = []
    res = None
    if w.op == "rms_norm":
        xbuf, x = _strided(d["x"], ldx, dt)
        rarn.rms_norm_ex(x, g, w.eps, out=y)
    else:
        rdt = w.res_dtype
        rbuf, res = _strided(d["residual"], ldr, rdt, extra=3)
        if w.op == "fused_add_rms_norm":
            xbuf, x = _strided(d["x"], ldx, dt)
            rarn.fused_add_rms_norm_ex(x, res, g, w.eps, out=y)
        else:
            R = w.R
            slice_ = T * ldx + pextra
            pbuf = torch.full((R * slice_,), FILL, dtype=g.dtype, device=g.device)
            for r in range(R):
                pbuf[r * slice_:r * slice_ + T * ldx].view(T, ldx)[:, :H].copy_(
                    to_device(d["partials"][r], dt))
            parts = pbuf.as_strided((R, T, H), (slice_, ldx, 1))
            rarn.reduce_add_rms_norm_ex(parts, res, g, w.eps, out=y)
        untouched.append(_padding_untouched(rbuf, T, H, ldr))
    torch.cuda.synchronize()
    untouched.append(_padding_untouched(ybuf, T, H, ldy))
    yb = to_host(y.contiguous(), dt)
    rb = None if res is None else to_host(res.contiguous(), w.res_dtype)
    return yb, rb, all(untouched)


def _oracle(w, d):
    """Oracle on the dense logical data (strides do not change the result:
    pinned on the CPU); the general form for a binary32 residual."""
    if w.res_dtype == w.dtype or w.op == "rms_norm":
        return run_oracle(w, d)
    T, H = w.T, w.H
    R = w.R if w.op == "reduce_add_rms_norm" else 1
    src = d["partials"] if w.op == "reduce_add_rms_norm" else d["x"][None]
    Y = np.zeros(T * H, d["gamma"].dtype)
    res = np.ascontiguousarray(d["residual"]).reshape(-1).copy()
    r = oracle.rows_ex(w.dtype, w.res_dtype, T, H, R, src.reshape(-1).copy(), H, T * H, res, H,
                       d["gamma"], w.eps, Y, H)
    r.y = r.y.reshape(T, H)
    r.residual = r.residual.reshape(T, H)
    return r


def _check(w, d, ldx, ldr, ldy, pextra=0, what=""):
    ref = _oracle(w, d)
    y, res, untouched = _run_strided(w, d, ldx, ldr, ldy, pextra)
    assert untouched, f"{what}: padding written"
    assert_y_close(y, ref.y, w.dtype, what)
    if res is not None:
        assert_bits_equal(res, ref.residual, what + " residual")


STRIDED = [  # T, H, ldx, ldr, ldy, partial-stride extra
    (33, 512, 576, 520, 600, 64),       # warp per row, 16-byte strides
    (5000, 512, 576, 512, 576, 0),      # many rows
    (3000, 4096, 4160, 4104, 4096, 8),  # pipelined CTA (plain / fused), stream (reduce)
    (17, 1000, 1003, 1001, 1005, 1),    # strides not 16-byte multiples: scalar
    (64, 16384, 16400, 16384, 16392, 0),
    (2000, 8192, 8200, 8192, 8200, 32),
]


@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"])
@pytest.mark.parametrize("dt", ["bf16", "f32", "f16"])
def test_strided_parity(op, dt):
    for T, H, ldx, ldr, ldy, pextra in STRIDED:
        if dt == "f32" and H * T > 20_000_000:
            continue
        w = W.workload(op, dt, T, H, R=3, eps=1e-6, seed=T + H)
        _check(w, W.generate(w), ldx, ldr, ldy, pextra, f"strided {op} {dt} T{T} H{H}")


@pytest.mark.parametrize("path", ["auto", "rows", "cluster", "stream"])
def test_strided_forced_paths(path):
    """Every kernel family with strided rows (where it runs the shape)."""
    for op, T, H, ld in (("fused_add_rms_norm", 3000, 4096, 4160),
                         ("reduce_add_rms_norm", 1000, 8192, 8264),
                         ("rms_norm", 64, 32768, 32832)):
        w = W.workload(op, "bf16", T, H, R=4, eps=1e-6, seed=T)
        rarn.set_path(path)
        if rarn.plan(op, T, H, 4, "bf16").startswith("none"):
            continue
        _check(w, W.generate(w), ld, ld + 8, ld + 16, 16, f"{path} {op}")


MIXED = [  # T, H: warp, pipelined CTA, single-wave CTA, cluster, scalar, two-pass
    (7, 64), (3000, 4096), (100, 5120), (64, 32768), (5, 1591), (3, 40000), (129, 8191),
]


@pytest.mark.parametrize("op", ["fused_add_rms_norm", "reduce_add_rms_norm"])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fp32_residual_parity(op, dt):
    for T, H in MIXED:
        w = W.workload(op, dt, T, H, R=3, eps=1e-6, seed=7 * T + H, rdtype="f32")
        assert w.res_dtype == "f32"
        _check(w, W.generate(w), H, H, H, 0, f"fp32 residual {op} {dt} T{T} H{H}")


@pytest.mark.parametrize("path", ["rows", "cluster"])
def test_fp32_residual_forced_paths(path):
    rarn.set_path(path)
    for op, T, H in (("fused_add_rms_norm", 64, 8192), ("reduce_add_rms_norm", 300, 4096)):
        w = W.workload(op, "bf16", T, H, R=2, eps=1e-6, seed=H, rdtype="f32")
        if rarn.plan(op, T, H, 2, "bf16", rdtype="f32").startswith("none"):
            continue
        _check(w, W.generate(w), H, H, H, 0, f"{path} fp32 residual {op}")


def test_fp32_residual_and_strides_together():
    w = W.workload("fused_add_rms_norm", "bf16", 2500, 4096, eps=1e-6, seed=3, rdtype="f32")
    _check(w, W.generate(w), 4160, 4100, 4104, 0, "fp32 residual + strides")


def test_stream_path_refuses_fp32_residual():
    rarn.set_path("stream")
    assert rarn.plan("fused_add_rms_norm", 5000, 4096, 1, "bf16", rdtype="f32").startswith("none")


@pytest.mark.parametrize("name", [w.name for w in W.EXTENDED])
def test_extended_workloads(name):
    """The widened rows' benchmark workloads at full size."""
    w = W.BY_NAME[name]
    _check(w, W.generate(w), w.row_stride, w.row_stride, w.row_stride, 0, name)


def test_fp32_residual_pipelined_warp():
    w = W.workload("fused_add_rms_norm", "bf16", 30000, 256, eps=1e-6, seed=5, rdtype="f32")
    assert "pipe=1" in rarn.plan(w.op, w.T, w.H, 1, "bf16", rdtype="f32")
    _check(w, W.generate(w), 256, 256, 256, 0, "fp32 residual warp pipe")
