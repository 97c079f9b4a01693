"""GPU parity of the reduce over 8-bit partials (e4m3 / e5m2 codes, one
binary32 scale per partial) against the CPU oracle: the updated residual
bit-exact, y within 2 ulps (binary32: 1e-5 relative), NaN where the oracle
has NaN."""
import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import assert_bits_equal, assert_y_close, to_device, to_host
from pins import lib_decode, lib_decode_fp8

pytestmark = pytest.mark.gpu

FMT_TOP = {"e4m3": 448.0, "e5m2": 57344.0}


def fp8in_inputs(R, T, H, dt, fmt, seed, scales=None, nan_codes=False):
    """Codes of finite values of both signs (N(0, 1) scaled to the format's
    range, rounded to codes with torch's float8 cast), per-partial scales,
    residual N(0, 1), gamma U(0.5, 1.5)."""
    import torch
    rng = np.random.default_rng(seed)
    td = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    v = rng.standard_normal((R, T, H)).astype(np.float32) * (FMT_TOP[fmt] / 16)
    codes = torch.from_numpy(v).to(td).view(torch.uint8).numpy()
    if nan_codes:
        codes[:, :, :3] = 0x7f  # NaN in both formats (e5m2: exponent all ones, mantissa 3)
    if scales is None:
        scales = rng.uniform(1e-3, 2.0, R).astype(np.float32)
    r = W.to_storage(rng.standard_normal((T, H)).astype(np.float32), dt)
    g = W.to_storage(rng.uniform(0.5, 1.5, H).astype(np.float32), dt)
    return codes, np.asarray(scales, np.float32), r, g


def run_fp8in(codes, scales, r, g, dt, fmt, eps=1e-6):
    import torch
    c = torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scales)).cuda()
    res = to_device(r, dt)
    y = rarn.reduce_add_rms_norm_fp8in(c, s, res, to_device(g, dt), eps, fmt)
    torch.cuda.synchronize()
    return to_host(y, dt), to_host(res, dt)


def check(codes, scales, r, g, dt, fmt, what, eps=1e-6, rows=None):
    y, res = run_fp8in(codes, scales, r, g, dt, fmt, eps)
    if rows is not None:
        codes, r, y, res = codes[:, rows], r[rows], y[rows], res[rows]
    want = oracle.reduce_fp8in(codes, scales, r, g, eps, dt, fmt)
    # residual: bit-exact, except that a NaN (from a NaN code) need only be a
    # NaN -- its payload is not specified
    nan_w = np.isnan(lib_decode(want.residual, dt))
    assert np.array_equal(np.isnan(lib_decode(res, dt)), nan_w), what + " residual NaNs"
    assert_bits_equal(np.where(nan_w, 0, res), np.where(nan_w, 0, want.residual),
                      what + " residual")
    assert_y_close(y, want.y, dt, what + " y")


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("R,T,H", [(1, 5, 8), (3, 37, 1592), (8, 64, 4096), (16, 9, 8192),
                                   (2, 300, 256), (5, 3, 16384)])
def test_fp8in_parity(dt, fmt, R, T, H):
    if dt == "f32" and H > 8192:
        pytest.skip("binary32 storage: H up to 8192")
    codes, scales, r, g = fp8in_inputs(R, T, H, dt, fmt, seed=R * 1000 + H + T)
    check(codes, scales, r, g, dt, fmt, f"{dt} {fmt} R{R} T{T} H{H}")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_fp8in_eight_element_packs(dt, tune):
    """The 8-element-pack kernel (the one H not a multiple of 16 takes)
    forced on shapes the 16-element kernel would take: same results."""
    tune(fp8in_pack16=0)
    for R, T, H, fmt in ((8, 40, 4096, "e4m3"), (3, 7, 8192, "e5m2")):
        codes, scales, r, g = fp8in_inputs(R, T, H, dt, fmt, seed=R + T + H)
        check(codes, scales, r, g, dt, fmt, f"8-element packs {dt} {fmt} R{R} H{H}")


def test_fp8in_power_of_two_scales_and_nan_codes():
    """Power-of-two scales (exact products), NaN codes (NaN rows in the
    residual and y), and a partial whose scale makes f16 overflow to inf."""
    R, T, H = 4, 6, 512
    codes, _, r, g = fp8in_inputs(R, T, H, "bf16", "e4m3", seed=7, nan_codes=True)
    check(codes, np.exp2([-3, 0, 2, 5]).astype(np.float32), r, g, "bf16", "e4m3",
          "pow2 scales, NaN codes")
    codes, _, r, g = fp8in_inputs(R, T, H, "f16", "e5m2", seed=8)
    check(codes, np.float32([4.0, 1.0, 1.0, 1.0]), r, g, "f16", "e5m2", "f16 overflow")


def test_fp8in_rejects():
    import torch
    c = torch.zeros(2, 4, 1004, dtype=torch.uint8, device="cuda")
    s = torch.ones(2, device="cuda")
    r = torch.zeros(4, 1004, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1004, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rarn.RarnError):
        rarn.reduce_add_rms_norm_fp8in(c, s, r, g, 1e-6)  # H = 1004: not a multiple of 8
    with pytest.raises(ValueError):
        rarn.reduce_add_rms_norm_fp8in(c, s[:1], r, g, 1e-6)


def test_fp8in_full_size_sampled():
    """The bench workload's shape (R = 8, bf16, [8192, 8192], e4m3), oracle on
    sampled rows."""
    R, T, H = 8, 8192, 8192
    codes, scales, r, g = fp8in_inputs(R, T, H, "bf16", "e4m3", seed=11)
    rows = np.linspace(0, T - 1, 48).astype(int)
    check(codes, scales, r, g, "bf16", "e4m3", "full size", rows=rows)


@pytest.mark.parametrize("R,T,H,kernel", [
    (4, 2048, 4096, "q8in.ring"),    # four partials, rows of 4096: the ring
    (3, 1300, 8192, "q8in.ring"),    # three partials, rows of 8192: the ring
    (6, 1300, 2048, "q8in.rows"),    # rows under 4096, fewer than 8 partials
])
def test_fp8in_planner_choice(R, T, H, kernel):
    """Shapes with at least 8 rows per SM that the planner sends to the ring
    or keeps on the register kernel by the partial count and row length:
    the plan says which, and the result matches the oracle on every row."""
    import torch
    props = torch.cuda.get_device_properties(0)
    if T < 8 * props.multi_processor_count:
        pytest.skip("fewer than 8 rows per SM on this device")
    smem = getattr(props, "shared_memory_per_block_optin", 0) or 232448
    plan = rarn.plan_fp8in(T, H, R, "bf16", True, props.multi_processor_count, smem)
    assert plan.startswith(kernel), plan
    codes, scales, r, g = fp8in_inputs(R, T, H, "bf16", "e4m3", seed=R * 31 + T)
    check(codes, scales, r, g, "bf16", "e4m3", f"R{R} T{T} H{H} ({kernel})")


@pytest.mark.parametrize("ring", [0, 1])
@pytest.mark.parametrize("pdl", [True, False])
def test_fp8in_chained(pdl, ring, tune):
    """Two dependent launches: the second reduces on the residual the first
    wrote (for the TMA-fed kernel, bulk copies of what the previous launch
    stored); replayed on the CPU with the oracle."""
    import torch
    tune(fp8in_ring=ring)
    rarn.set_pdl(pdl)
    try:
        R, T, H = 3, 40, 2048
        codes, scales, r, g = fp8in_inputs(R, T, H, "bf16", "e4m3", seed=12)
        c = torch.from_numpy(codes).cuda()
        s = torch.from_numpy(scales).cuda()
        res = to_device(r, "bf16")
        gd = to_device(g, "bf16")
        rarn.reduce_add_rms_norm_fp8in(c, s, res, gd, 1e-6)
        y2 = rarn.reduce_add_rms_norm_fp8in(c, s, res, gd, 1e-6)
        torch.cuda.synchronize()
        o1 = oracle.reduce_fp8in(codes, scales, r, g, 1e-6, "bf16", "e4m3")
        o2 = oracle.reduce_fp8in(codes, scales, o1.residual, g, 1e-6, "bf16", "e4m3")
        assert_bits_equal(to_host(res, "bf16"), o2.residual, "chained residual")
        assert_y_close(to_host(y2, "bf16"), o2.y, "bf16", "chained y")
    finally:
        rarn.set_pdl(True)


def all_finite_codes(fmt):
    """Every finite code of the format (both zeros, subnormals, normals)."""
    c = np.arange(256, dtype=np.uint8)
    special = (c & 0x7F) == 0x7F if fmt == "e4m3" else (c & 0x7C) == 0x7C
    return c[~special]


def test_fp8in_tma_fed_kernel(tune):
    """The TMA-fed kernel forced on shapes the register kernels would take:
    ragged last chunks, 1 to 16 partials, all three storage types, every
    finite code, NaN and Inf codes, and overflow of the sum."""
    tune(fp8in_ring=1)
    for dt, fmt, R, T, H in (("bf16", "e4m3", 8, 40, 4096), ("f16", "e5m2", 3, 37, 1040),
                             ("f32", "e4m3", 5, 9, 8192), ("bf16", "e5m2", 16, 5, 16384),
                             ("bf16", "e4m3", 2, 300, 16), ("f16", "e4m3", 1, 11, 6144),
                             ("f32", "e5m2", 4, 160, 2064)):
        codes, scales, r, g = fp8in_inputs(R, T, H, dt, fmt, seed=R * 7 + T + H)
        check(codes, scales, r, g, dt, fmt, f"tma-fed {dt} {fmt} R{R} T{T} H{H}")
    for fmt in ("e4m3", "e5m2"):
        fin = all_finite_codes(fmt)
        R, T, H = 3, 6, 512
        codes = np.stack([np.resize(np.roll(fin, 17 * k + t), H) for k in range(R)
                          for t in range(T)]).reshape(R, T, H)
        _, _, r, g = fp8in_inputs(R, T, H, "bf16", fmt, seed=21)
        check(codes, np.float32([1.0, 0.37, 2.0 ** -10]), r, g, "bf16", fmt,
              f"tma-fed every finite {fmt} code")
    codes, _, r, g = fp8in_inputs(4, 6, 512, "bf16", "e4m3", seed=7, nan_codes=True)
    check(codes, np.exp2([-3, 0, 2, 5]).astype(np.float32), r, g, "bf16", "e4m3",
          "tma-fed NaN codes")
    codes, _, r, g = fp8in_inputs(4, 6, 512, "f16", "e5m2", seed=8)
    codes[1, :, 5] = 0x7C  # +Inf
    codes[2, 2, 9] = 0xFC  # -Inf
    check(codes, np.float32([4.0, 1.0, 1.0, 1.0]), r, g, "f16", "e5m2",
          "tma-fed Inf codes, f16 overflow")


@pytest.mark.parametrize("fill", [0, 3])
def test_fp8in_wait_runs_out_and_is_reported(fill, tune):
    """Failure detection without a GPU fault: the TMA-fed kernel's test hook
    leaves one ring fill of CTA 0 without its last 16 bytes; the consumers'
    wait gives up after 20 ms, the CTA drains its copies and returns, the
    watchdog bit is set, and the next call is correct."""
    import torch
    tune(fp8in_ring=1)
    rarn.watchdog(clear=True)
    R, T, H = 4, 1000, 4096  # CTA 0 takes 7 rows, one fill each
    codes, scales, r, g = fp8in_inputs(R, T, H, "bf16", "e4m3", seed=30 + fill)
    assert rarn.library().rarn_test_stall(fill, 20_000_000) == 0
    run_fp8in(codes, scales, r, g, "bf16", "e4m3")  # outputs not valid; the call returns
    torch.cuda.synchronize()
    flags = rarn.watchdog(clear=True)
    assert flags & 1, f"consumer timeout not reported (flags={flags})"
    check(codes, scales, r, g, "bf16", "e4m3", "after a watchdog timeout")
    assert rarn.watchdog(clear=True) == 0
