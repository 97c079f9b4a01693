"""GPU parity: the CUDA library against the CPU oracle, element by element.

Every configuration of the method at its full size, an edge-shape grid,
unaligned and in-place buffers, guard bands around the outputs, determinism,
and the stored golden fixture.  Residual bit-exact; y within 1e-5 relative
(fp32) or 2 ulps (fp16 / bf16).
"""
import functools

import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import (assert_bits_equal, assert_y_close, check_parity, run_gpu, run_oracle,
                      to_device, to_host)

pytestmark = pytest.mark.gpu

PATHS = ["auto", "rows", "stream", "cluster"]


@pytest.fixture(autouse=True)
def _reset_path():
    yield
    rarn.set_path("auto")


def _supported(w, path):
    """Whether a forced path can run this shape (auto always can)."""
    rarn.set_path(path)
    R = w.R if w.op == "reduce_add_rms_norm" else 0
    text = rarn.plan(w.op, w.T, w.H, max(R, 1), w.dtype)
    return not text.startswith("none")


@functools.lru_cache(maxsize=1)
def _config_data(name):
    w = W.BY_NAME[name]
    d = W.generate(w)
    return w, d, run_oracle(w, d)


CONFIG_CASES = [(w.name, p) for w in W.CONFIGS for p in PATHS]


@pytest.mark.parametrize("name,path", CONFIG_CASES, ids=[f"{n}-{p}" for n, p in CONFIG_CASES])
def test_config_parity(name, path):
    w, d, ref = _config_data(name)
    if not _supported(w, path):
        pytest.skip(f"path {path} does not run {name}")
    rarn.set_path(path)
    y, res = run_gpu(w, d)
    assert_y_close(y, ref.y, w.dtype, f"{name}/{path}")
    if ref.residual is not None:
        assert_bits_equal(res, ref.residual, f"{name}/{path} residual")


EDGE_H = [1, 7, 8, 9, 31, 33, 127, 1591, 1592, 1593, 4095, 5120, 8191, 16384, 16385]
EDGE_T = [1, 2, 3, 131]


def _edge_cases():
    cases = []
    for dt in ("f32", "f16", "bf16"):
        for H in EDGE_H:
            for T in EDGE_T:
                if T == 131 and H > 5120 and dt != "bf16":
                    continue
                cases.append(("rms_norm", dt, T, H, 0))
                cases.append(("fused_add_rms_norm", dt, T, H, 1))
                for R in ((2, 3, 8) if H <= 1593 else (3,)):
                    cases.append(("reduce_add_rms_norm", dt, T, H, R))
    return cases


EDGE = _edge_cases()


@pytest.mark.parametrize("path", PATHS)
def test_edge_grid(path):
    """All edge shapes under one forced path (skipping shapes it cannot run)."""
    ran = 0
    for op, dt, T, H, R in EDGE:
        w = W.workload(op, dt, T, H, R=R, eps=1e-5, seed=T * 100003 + H)
        if not _supported(w, path):
            continue
        rarn.set_path(path)
        check_parity(w, W.generate(w), what=f"{op}/{dt}/T{T}/H{H}/R{R}/{path}")
        ran += 1
    if path in ("auto", "rows"):
        assert ran == len(EDGE)
    elif ran == 0:
        pytest.skip(f"path {path} runs none of the edge shapes")


@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place_output(op, dt):
    """y may overwrite x (or partial 0)."""
    for H in (1592, 4096, 5121):
        w = W.workload(op, dt, 37, H, eps=1e-6, seed=H)
        check_parity(w, W.generate(w), out_is_input=True, what=f"in-place {op} {dt} H{H}")


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_unaligned_pointers(dt):
    """Buffers offset by one element from a 16-byte boundary run the scalar
    kernels and give the same results."""
    import torch
    T, H = 19, 1024
    for op in ("rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"):
        w = W.workload(op, dt, T, H, R=3, eps=1e-6, seed=5)
        d = W.generate(w)
        ref = run_oracle(w, d)

        def shifted(bits):
            t = to_device(bits.reshape(-1), dt)
            buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
            v = buf[1:]
            v.copy_(t)
            return v

        g = shifted(d["gamma"])
        y = shifted(np.zeros((T, H), d["gamma"].dtype)).view(T, H)
        if op == "rms_norm":
            rarn.rms_norm(shifted(d["x"]).view(T, H), g, w.eps, out=y)
            res = None
        elif op == "fused_add_rms_norm":
            res = shifted(d["residual"]).view(T, H)
            rarn.fused_add_rms_norm(shifted(d["x"]).view(T, H), res, g, w.eps, out=y)
        else:
            res = shifted(d["residual"]).view(T, H)
            p = shifted(d["partials"]).view(3, T, H)
            rarn.reduce_add_rms_norm(p, res, g, w.eps, out=y)
        torch.cuda.synchronize()
        assert_y_close(to_host(y, dt), ref.y, dt, f"unaligned {op}")
        if res is not None:
            assert_bits_equal(to_host(res, dt), ref.residual, f"unaligned {op} residual")


@pytest.mark.parametrize("path", PATHS)
def test_guard_bands(path):
    """Nothing is written outside y and the residual: 256-byte guards on both
    sides keep their pattern."""
    import torch
    G = 128  # bf16 elements = 256 bytes
    for op, T, H in (("fused_add_rms_norm", 133, 4096), ("reduce_add_rms_norm", 61, 5120),
                     ("rms_norm", 300, 1000), ("fused_add_rms_norm", 7, 16385)):
        w = W.workload(op, "bf16", T, H, R=4, eps=1e-6, seed=9)
        if not _supported(w, path):
            continue
        rarn.set_path(path)
        d = W.generate(w)
        ref = run_oracle(w, d)

        def guarded(bits):
            t = to_device(bits.reshape(-1), "bf16")
            buf = torch.full((t.numel() + 2 * G,), -7.0, dtype=t.dtype, device=t.device)
            buf[G:G + t.numel()].copy_(t)
            return buf

        ybuf = guarded(np.zeros(T * H, np.uint16))
        y = ybuf[G:G + T * H].view(T, H)
        g = to_device(d["gamma"], "bf16")
        rbuf = None
        if op == "rms_norm":
            rarn.rms_norm(to_device(d["x"], "bf16"), g, w.eps, out=y)
        else:
            rbuf = guarded(d["residual"])
            res = rbuf[G:G + T * H].view(T, H)
            if op == "fused_add_rms_norm":
                rarn.fused_add_rms_norm(to_device(d["x"], "bf16"), res, g, w.eps, out=y)
            else:
                rarn.reduce_add_rms_norm(to_device(d["partials"], "bf16"), res, g, w.eps, out=y)
        torch.cuda.synchronize()
        for buf in (ybuf, rbuf):
            if buf is None:
                continue
            assert torch.all(buf[:G] == -7.0) and torch.all(buf[G + T * H:] == -7.0), \
                f"guard overwritten: {op} {path}"
        assert_y_close(to_host(y, "bf16"), ref.y, "bf16", f"guarded {op}")
        if rbuf is not None:
            assert_bits_equal(to_host(rbuf[G:G + T * H], "bf16").reshape(T, H), ref.residual)


def test_deterministic_bits():
    """Two runs on the same inputs give identical bits, every path."""
    w = W.BY_NAME["fused_bf16_T4096_H4096"]
    d = W.generate(w)
    for path in PATHS:
        if not _supported(w, path):
            continue
        rarn.set_path(path)
        a = run_gpu(w, d)
        b = run_gpu(w, d)
        assert_bits_equal(a[0], b[0], f"y {path}")
        assert_bits_equal(a[1], b[1], f"residual {path}")


def test_zero_row_with_zero_eps_gives_nan():
    """A zero row with eps = 0: inv = +inf and y = 0 * inf = NaN, as in the
    oracle."""
    w = W.workload("rms_norm", "f32", 4, 64, eps=0.0)
    d = W.generate(w)
    d["x"][2] = 0.0
    y, _ = run_gpu(w, d)
    ref = run_oracle(w, d)
    assert np.all(np.isnan(ref.y[2])) and np.all(np.isnan(y[2]))
    assert_y_close(y, ref.y, "f32")


def test_many_rows_grid_stride():
    """T far above the grid size: every row is visited exactly once."""
    for op, dt, T, H in (("rms_norm", "bf16", 200003, 64), ("fused_add_rms_norm", "f16", 50001,
                                                            1024),
                         ("reduce_add_rms_norm", "bf16", 20011, 2048)):
        w = W.workload(op, dt, T, H, R=2, eps=1e-6, seed=3)
        check_parity(w, W.generate(w), what=f"grid-stride {op}")


def test_golden_fixture_on_gpu():
    """The stored oracle outputs (tests/golden/oracle_small.json)."""
    from golden_io import cases
    for c in cases():
        w = W.workload(c["op"], c["dtype"], c["T"], c["H"], R=c["R"], eps=c["eps"])
        y, res = run_gpu(w, c["inputs"])
        assert_y_close(y, c["expected"]["y"], c["dtype"], f"golden {c['op']} {c['dtype']}")
        if "residual" in c["expected"]:
            assert_bits_equal(res, c["expected"]["residual"], "golden residual")


def test_binding_rejects_bad_tensors():
    import torch
    x = torch.zeros(4, 8, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(8, device="cuda", dtype=torch.float16)
    with pytest.raises(TypeError):
        rarn.rms_norm(x, g, 1e-6)
    with pytest.raises(ValueError):
        rarn.rms_norm(x.t(), torch.ones(4, device="cuda", dtype=torch.bfloat16), 1e-6)
    with pytest.raises(rarn.RarnError):
        rarn.fused_add_rms_norm(x, x, torch.ones(8, device="cuda", dtype=torch.bfloat16), 1e-6)


def test_watchdog_clear_after_everything():
    assert rarn.watchdog(clear=True) == 0


@pytest.mark.parametrize("ppt", [1, 2, 4])
@pytest.mark.parametrize("groups", [1, 2])
def test_stream_consumer_groups(groups, ppt, tune):
    """The TMA-fed kernel with 1 and 2 consumer groups (rows handed out
    round-robin) and 1, 2, 4 packs per thread per chunk, including row
    counts that are not a multiple of the grid times the group count, and
    rows of one, several and a partial chunk."""
    tune(stream_groups=groups, stream_packs=ppt)
    rarn.set_path("stream")
    for op, dt, T, H, R in (("fused_add_rms_norm", "bf16", 1001, 4096, 1),
                            ("reduce_add_rms_norm", "bf16", 777, 2048, 8),
                            ("reduce_add_rms_norm", "f16", 333, 5120, 3),
                            ("rms_norm", "f32", 999, 1592, 0),
                            ("fused_add_rms_norm", "bf16", 157, 32768, 1),
                            ("fused_add_rms_norm", "f32", 5, 200, 1)):
        w = W.workload(op, dt, T, H, R=R, eps=1e-6, seed=groups * 10 + ppt)
        plan = rarn.plan(op, T, H, max(R, 1), dt)
        assert plan.startswith("stream"), plan
        check_parity(w, W.generate(w), what=f"stream G{groups} {op} {dt} T{T} H{H}")


def _pinned(bits, dt):
    import torch
    if dt == "f32":
        t = torch.from_numpy(np.ascontiguousarray(bits, np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
        t = t.view({"f16": torch.float16, "bf16": torch.bfloat16}[dt])
    return t.pin_memory()


@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm", "reduce_add_rms_norm"])
def test_host_buffers(op):
    """The *_host entry points on pinned host memory: the kernels read and
    write the host buffers through their device mapping; same results."""
    import torch
    for dt, T, H in (("bf16", 300, 4096), ("f32", 7, 1593), ("f16", 129, 8192),
                     ("bf16", 3, 40000)):
        w = W.workload(op, dt, T, H, R=3, eps=1e-6, seed=T + H)
        d = W.generate(w)
        ref = run_oracle(w, d)
        g = _pinned(d["gamma"], dt)
        if op == "rms_norm":
            y = rarn.rms_norm_host(_pinned(d["x"], dt), g, w.eps)
            res = None
        elif op == "fused_add_rms_norm":
            res = _pinned(d["residual"], dt)
            y = rarn.fused_add_rms_norm_host(_pinned(d["x"], dt), res, g, w.eps)
        else:
            res = _pinned(d["residual"], dt)
            y = rarn.reduce_add_rms_norm_host(_pinned(d["partials"], dt), res, g, w.eps)
        torch.cuda.synchronize()
        assert_y_close(to_host(y, dt), ref.y, dt, f"host {op} {dt} T{T} H{H}")
        if res is not None:
            assert_bits_equal(to_host(res, dt), ref.residual, f"host {op} residual")


def test_host_buffers_memory_kinds():
    """Pageable host memory is used where the device reads it through the
    host's page tables (rarn_host_access() == 2, e.g. Grace) and refused
    otherwise; device memory is always refused; nothing is launched on a
    refusal (the output keeps its contents)."""
    import ctypes

    import torch
    lib = rarn.library()
    access = lib.rarn_host_access()
    assert access in (1, 2)
    x = torch.full((4, 64), 2.0, dtype=torch.bfloat16)    # pageable
    g = torch.ones(64, dtype=torch.bfloat16).pin_memory()
    y = torch.zeros(4, 64, dtype=torch.bfloat16).pin_memory()
    st = lib.rarn_rms_norm_host(y.data_ptr(), x.data_ptr(), g.data_ptr(), 4, 64, 1e-6, 2,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    if access == 2:
        assert st == 0
        assert torch.allclose(y.float(), torch.ones(4, 64), rtol=0, atol=1e-2)
    else:
        assert st == 1  # RARN_ERR_INVALID_ARG
    xd = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    y.fill_(5.0)
    st = lib.rarn_rms_norm_host(y.data_ptr(), xd.data_ptr(), g.data_ptr(), 4, 64, 1e-6, 2,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 1
    assert torch.all(y == 5.0)
    with pytest.raises(ValueError):
        rarn.rms_norm_host(x, g, 1e-6)  # the binding asks for pinned tensors
    torch.cuda.synchronize()


@pytest.mark.parametrize("pdl", [False, True])
def test_chained_launches(pdl):
    """Three launches in a row on one stream, each reading what the previous
    one wrote (y becomes the next x; the residual carries over), with and
    without programmatic dependent launch: each step matches the oracle run
    on that step's actual inputs (the GPU's y of the step before)."""
    import torch
    rarn.set_pdl(pdl)
    try:
        for path, T, H in (("auto", 4096, 4096), ("stream", 2000, 8192), ("rows", 3, 5120),
                           ("cluster", 64, 32768)):
            w = W.workload("fused_add_rms_norm", "bf16", T, H, eps=1e-6, seed=T)
            if not _supported(w, path):
                continue
            rarn.set_path(path)
            d = W.generate(w)
            x = to_device(d["x"], "bf16")
            res = to_device(d["residual"], "bf16")
            g = to_device(d["gamma"], "bf16")
            bufs = [torch.empty_like(x) for _ in range(3)]
            cur = x
            for b in bufs:
                rarn.fused_add_rms_norm(cur, res, g, w.eps, out=b)
                cur = b
            torch.cuda.synchronize()
            xs, rs = d["x"], d["residual"]
            for k in range(3):
                ref = oracle.fused_add_rms_norm(xs, rs, d["gamma"], w.eps, "bf16")
                yk = to_host(bufs[k], "bf16")
                assert_y_close(yk, ref.y, "bf16", f"chain step {k} {path} pdl={pdl}")
                xs, rs = yk, ref.residual
            assert_bits_equal(to_host(res, "bf16"), rs, f"chain residual {path} pdl={pdl}")
    finally:
        rarn.set_pdl(True)
        rarn.set_path("auto")


def test_pipelined_rows_kernel():
    """The software-pipelined CTA kernel (next row's loads issued before the
    current row is reduced and written): several rows per CTA, ragged row
    counts, and y written over x in place."""
    for op, dt, T, H, inplace in (("fused_add_rms_norm", "bf16", 5003, 2048, False),
                                  ("rms_norm", "f32", 3001, 4096, False),
                                  ("fused_add_rms_norm", "f16", 7777, 1600, True),
                                  ("rms_norm", "bf16", 9000, 3000, True),
                                  ("fused_add_rms_norm", "bf16", 40000, 5120, False),
                                  ("fused_add_rms_norm", "bf16", 4099, 16384, False)):
        w = W.workload(op, dt, T, H, eps=1e-6, seed=T)
        plan = rarn.plan(op, T, H, 1, dt)
        assert "pipe=1" in plan, plan
        check_parity(w, W.generate(w), out_is_input=inplace, what=f"pipe {op} {dt} T{T} H{H}")


def test_pipelined_warp_kernel():
    """The pipelined warp-per-row kernel: short rows, several rows per warp,
    ragged row counts, in place."""
    for op, dt, T, H, inplace in (("rms_norm", "f32", 20011, 96, False),
                                  ("fused_add_rms_norm", "bf16", 30001, 1024, True),
                                  ("rms_norm", "f16", 25000, 512, True),
                                  ("fused_add_rms_norm", "f16", 10999, 8, False)):
        w = W.workload(op, dt, T, H, eps=1e-6, seed=T)
        plan = rarn.plan(op, T, H, 1, dt)
        assert plan.startswith("rows.warp") and "pipe=1" in plan, plan
        check_parity(w, W.generate(w), out_is_input=inplace, what=f"warp pipe {op} {dt} T{T}")
