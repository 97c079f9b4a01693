"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, rejects bad arguments before touching a GPU, and plans kernels.
CPU only: no call here launches anything."""
import ctypes
import os
import re

import pytest

import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import build as rbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "rarn.h")

OK, INVALID, UNSUPPORTED, ALIAS, CUDA = 0, 1, 2, 3, 4
F32, F16, BF16 = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return rarn.library()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rarn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.rarn_version() >> 16 == 1
    for code in range(5):
        assert lib.rarn_status_string(code)
    assert lib.rarn_status_string(99) == b"unknown status"


# fake, never dereferenced device addresses: argument checks run before any
# CUDA call, so these calls never reach the GPU
A, B, C, D = 1 << 40, 2 << 40, 3 << 40, 4 << 40


@pytest.mark.parametrize("args,want", [
    ((A, B, C, 4, 0, 1e-6, BF16, None), INVALID),        # H = 0
    ((A, B, C, -1, 8, 1e-6, BF16, None), INVALID),       # T < 0
    ((A, B, C, 4, 8, -1.0, BF16, None), INVALID),        # eps < 0
    ((A, B, C, 4, 8, float("nan"), BF16, None), INVALID),
    ((A, B, C, 4, 8, float("inf"), BF16, None), INVALID),
    ((A, B, C, 4, 8, 1e-6, 7, None), INVALID),           # dtype
    ((None, B, C, 4, 8, 1e-6, BF16, None), INVALID),     # null y
    ((A, None, C, 4, 8, 1e-6, BF16, None), INVALID),     # null x
    ((A, B, None, 4, 8, 1e-6, BF16, None), INVALID),     # null gamma
    ((A, B, C, 4, (1 << 24) + 1, 1e-6, BF16, None), UNSUPPORTED),
    ((A, A + 2, C, 4, 8, 1e-6, BF16, None), ALIAS),      # y overlaps x, not equal
    ((A, B, A + 16, 4, 8, 1e-6, BF16, None), ALIAS),     # gamma inside y
    ((None, None, None, 0, 8, 1e-6, BF16, None), OK),    # T = 0 is a no-op
])
def test_rms_norm_argument_errors(lib, args, want):
    assert lib.rarn_rms_norm(*args) == want


@pytest.mark.parametrize("args,want", [
    ((A, B, None, D, 4, 8, 1e-6, F16, None), INVALID),   # null residual
    ((A, B, A, D, 4, 8, 1e-6, F16, None), ALIAS),        # residual == y
    ((A, B, B, D, 4, 8, 1e-6, F16, None), ALIAS),        # residual == x
    ((A, B, C, C + 8, 4, 8, 1e-6, F16, None), ALIAS),    # gamma inside residual
    ((A, B, C, D, 0, 8, 1e-6, F16, None), OK),
])
def test_fused_argument_errors(lib, args, want):
    assert lib.rarn_fused_add_rms_norm(*args) == want


@pytest.mark.parametrize("args,want", [
    ((A, B, 0, C, D, 4, 8, 1e-6, F32, None), INVALID),   # R = 0
    ((A, B, 65, C, D, 4, 8, 1e-6, F32, None), UNSUPPORTED),  # R > max
    # y == partial 0 is allowed, but y overlapping partial 1 is not
    ((B + 4 * 8 * 4, B, 2, C, D, 4, 8, 1e-6, F32, None), ALIAS),
    # residual inside partial 2
    ((A, B, 3, B + 2 * 4 * 8 * 4, D, 4, 8, 1e-6, F32, None), ALIAS),
    ((A, B, 8, C, D, 0, 8, 1e-6, F32, None), OK),
])
def test_reduce_argument_errors(lib, args, want):
    assert lib.rarn_reduce_add_rms_norm(*args) == want


def test_path_setting(lib):
    assert rarn.get_path() == "auto"
    for name in ("rows", "stream", "cluster", "auto"):
        rarn.set_path(name)
        assert rarn.get_path() == name
    assert lib.rarn_set_path(9) == INVALID
    assert rarn.get_path() == "auto"


def test_watchdog_null_pointer(lib):
    assert lib.rarn_watchdog(None, 0) == INVALID


def _plan(op, T, H, R, dt, vec=True):
    return rarn.plan(op, T, H, R, dt, vec_ok=vec, num_sms=152)


def test_plan_rows_kinds():
    rarn.set_path("rows")
    try:
        # short rows: a warp per row
        assert _plan("rms_norm", 512, 512, 0, "bf16").startswith("rows.warp")
        assert _plan("rms_norm", 512, 1024, 0, "bf16").startswith("rows.warp")
        # medium rows: a CTA per row, packs
        p = _plan("fused_add_rms_norm", 4096, 4096, 1, "bf16")
        assert p.startswith("rows.cta vec16"), p
        # H*2 bytes not a multiple of 16: scalar kernel
        assert "scalar" in _plan("fused_add_rms_norm", 8, 1591, 1, "bf16")
        # unaligned pointers: scalar kernel
        assert "scalar" in _plan("fused_add_rms_norm", 8, 4096, 1, "bf16", vec=False)
        # rows beyond the register budget: two passes
        assert _plan("fused_add_rms_norm", 8, 1 << 20, 1, "bf16").startswith("rows.two_pass")
        assert _plan("rms_norm", 8, 20000, 0, "f16", vec=False).startswith("rows.two_pass")
    finally:
        rarn.set_path("auto")


def test_plan_grid_is_capped_and_covers_small_t():
    rarn.set_path("rows")
    try:
        p = _plan("fused_add_rms_norm", 3, 4096, 1, "bf16")
        assert "grid=3 " in p, p
        p = _plan("fused_add_rms_norm", 1 << 20, 4096, 1, "bf16")
        grid = int(re.search(r"grid=(\d+)", p).group(1))
        assert grid <= 152 * 8, p
    finally:
        rarn.set_path("auto")


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(rarn, "_lib", None)
    monkeypatch.setattr(rarn, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        rarn.library()


def test_header_declares_three_compute_calls():
    names = declared_functions()
    for n in ("rarn_rms_norm", "rarn_fused_add_rms_norm", "rarn_reduce_add_rms_norm"):
        assert n in names


def test_plan_auto_policy():
    """The automatic choice per shape (152 SMs)."""
    assert rarn.get_path() == "auto"
    # R = 8 reduce at full size: the TMA-fed stream kernel, one consumer group
    p = _plan("reduce_add_rms_norm", 8192, 8192, 8, "bf16")
    assert p.startswith("stream") and "groups=1" in p, p
    # R = 2 reduce: stream kernel with two consumer groups
    p = _plan("reduce_add_rms_norm", 16384, 4096, 2, "bf16")
    assert p.startswith("stream") and "groups=2" in p, p
    # fused / plain rows that fit one CTA's registers: the pipelined register
    # kernel; longer rows: the stream kernel
    for H in (4096, 8192, 16384):
        p = _plan("fused_add_rms_norm", 4096, H, 1, "bf16")
        assert p.startswith("rows.cta") and "pipe=1" in p, p
    assert _plan("fused_add_rms_norm", 4096, 32768, 1, "bf16").startswith("stream")
    p = _plan("rms_norm", 4096, 20000, 0, "bf16")
    assert p.startswith("stream") and "groups=2" in p, p
    # few rows: never the persistent kernel
    assert _plan("reduce_add_rms_norm", 64, 8192, 8, "bf16").startswith("rows")
    # 32 KB rows, few of them: one CTA per row still holds the row (one row
    # per SM at most: as many threads as the register budget allows, 512 of 4
    # packs); 64 KB rows need a cluster per row
    p = _plan("fused_add_rms_norm", 64, 16384, 1, "bf16")
    assert p.startswith("rows.cta") and "per_thread=4 block=512" in p, p
    # one wave of rows: up to 1024 threads per row; more rows than SMs: 256
    assert "per_thread=1 block=640" in _plan("fused_add_rms_norm", 128, 5120, 1, "bf16")
    assert "per_thread=1 block=1024" in _plan("rms_norm", 152, 8192, 0, "bf16")
    assert "per_thread=4 block=160" in _plan("fused_add_rms_norm", 153, 5120, 1, "bf16")
    assert "per_thread=2 block=256" in _plan("reduce_add_rms_norm", 64, 4096, 8, "bf16")
    p = _plan("fused_add_rms_norm", 64, 32768, 1, "bf16")
    assert p.startswith("cluster"), p
    # a single wave keeps gamma in registers; many rounds read it from L1
    assert "gamma_regs=1" in _plan("fused_add_rms_norm", 16, 5120, 1, "bf16")
    assert "gamma_regs=0" in _plan("fused_add_rms_norm", 32768, 5120, 1, "bf16")
    # balanced grid: 4096 rows on 1216 slots -> 4 rounds of 1024 CTAs
    assert "grid=1024 " in _plan("fused_add_rms_norm", 4096, 4096, 1, "bf16")
    # unaligned: scalar register kernels whatever the size
    assert "scalar" in _plan("reduce_add_rms_norm", 8192, 8192, 8, "bf16", vec=False)
    # plain: register kernel
    assert _plan("rms_norm", 16384, 4096, 0, "bf16").startswith("rows.cta")


def test_pdl_setting_and_stall_hook_arguments(lib):
    assert rarn.get_pdl() is True  # on by default
    rarn.set_pdl(False)
    assert rarn.get_pdl() is False
    rarn.set_pdl(True)
    assert rarn.get_pdl() is True
    assert lib.rarn_test_stall(-1, 1000) == INVALID
    assert lib.rarn_test_stall(0, 0) == INVALID
    assert lib.rarn_test_stall(0, 3_000_000_000) == INVALID


def _rows(ptr, ld, dt):
    return rarn.Rows(ptr, ld, dt)


def test_general_forms_argument_errors(lib):
    """General forms: storage-type combinations, strides and aliasing are
    checked before any CUDA call."""
    H, T = 64, 4
    # residual f16 with bf16 inputs: not a supported combination
    st = lib.rarn_fused_add_rms_norm_ex(_rows(A, H, BF16), _rows(B, H, BF16), _rows(C, H, F16), D,
                                        T, H, 1e-6, None)
    assert st == UNSUPPORTED
    # fp32 inputs with a 16-bit residual: not supported either
    st = lib.rarn_fused_add_rms_norm_ex(_rows(A, H, F32), _rows(B, H, F32), _rows(C, H, BF16), D,
                                        T, H, 1e-6, None)
    assert st == UNSUPPORTED
    # y of another type than x
    assert lib.rarn_rms_norm_ex(_rows(A, H, F16), _rows(B, H, BF16), D, T, H, 1e-6,
                                None) == UNSUPPORTED
    # row stride below H
    assert lib.rarn_rms_norm_ex(_rows(A, H, BF16), _rows(B, H - 1, BF16), D, T, H, 1e-6,
                                None) == INVALID
    # y interleaved with x inside one allocation: spans overlap -> refused
    assert lib.rarn_rms_norm_ex(_rows(A + 2 * H, 2 * H, BF16), _rows(A, 2 * H, BF16), D, T, H,
                                1e-6, None) == ALIAS
    # in place with the same stride is allowed (fails later only for lack of a GPU)
    st = lib.rarn_rms_norm_ex(_rows(A, 2 * H, BF16), _rows(A, 2 * H, BF16), D, T, H, 1e-6, None)
    assert st not in (INVALID, ALIAS, UNSUPPORTED)
    # residual inside the span of partial 1 (partials 10 000 elements apart)
    st = lib.rarn_reduce_add_rms_norm_ex(_rows(A, H, BF16), _rows(B, H, BF16), 10000, 2,
                                         _rows(B + 2 * 10000 + 8, H, F32), D, T, H, 1e-6, None)
    assert st == ALIAS
    # T = 0 is a no-op whatever the pointers
    assert lib.rarn_rms_norm_ex(_rows(None, H, BF16), _rows(None, H, BF16), None, 0, H, 1e-6,
                                None) == OK


def test_plan_fp32_residual():
    p = rarn.plan("fused_add_rms_norm", 32768, 5120, 1, "bf16", num_sms=152, rdtype="f32")
    assert p.startswith("rows.cta") and "pipe=1" in p, p
    # the stream kernel is for one storage type only: a long fp32-residual row
    # with many rows goes to the two-pass / cluster kernels
    p = rarn.plan("fused_add_rms_norm", 4096, 40000, 1, "bf16", num_sms=152, rdtype="f32")
    assert not p.startswith("stream"), p
    assert rarn.plan("fused_add_rms_norm", 8, 4096, 1, "f32", num_sms=152, rdtype="bf16") \
        .startswith("none")


def _fp8(ptr, ld, fmt=0, mode=0, scale=C + (1 << 30)):
    return ctypes.byref(rarn.Fp8Rows(ptr, ld, fmt, mode, scale))


def test_fp8_forms_argument_errors(lib):
    """8-bit output forms: descriptor, storage types and aliasing are checked
    before any CUDA call."""
    H, T = 64, 4
    x = _rows(B, H, BF16)
    assert lib.rarn_rms_norm_fp8(None, x, D, T, H, 1e-6, None) == INVALID
    assert lib.rarn_rms_norm_fp8(_fp8(A, H, fmt=2), x, D, T, H, 1e-6, None) == INVALID
    assert lib.rarn_rms_norm_fp8(_fp8(A, H, mode=2), x, D, T, H, 1e-6, None) == INVALID
    assert lib.rarn_rms_norm_fp8(_fp8(A, H, scale=None), x, D, T, H, 1e-6, None) == INVALID
    assert lib.rarn_rms_norm_fp8(_fp8(A, H - 1), x, D, T, H, 1e-6, None) == INVALID
    # an fp32 residual with 16-bit inputs is not built for the 8-bit output
    st = lib.rarn_fused_add_rms_norm_fp8(_fp8(A, H), x, _rows(C, H, F32), D, T, H, 1e-6, None)
    assert st == UNSUPPORTED
    # codes over x; per-row scales inside x; per-tensor scale inside the codes
    assert lib.rarn_rms_norm_fp8(_fp8(B + 8, H), x, D, T, H, 1e-6, None) == ALIAS
    assert lib.rarn_rms_norm_fp8(_fp8(A, H, mode=1, scale=B + 16), x, D, T, H, 1e-6,
                                 None) == ALIAS
    assert lib.rarn_rms_norm_fp8(_fp8(A, H, mode=0, scale=A + 4), x, D, T, H, 1e-6,
                                 None) == ALIAS
    # a per-tensor scale may sit inside an input (it is only read) ...
    st = lib.rarn_rms_norm_fp8(_fp8(A, H, mode=0, scale=B + 16), x, D, T, H, 1e-6, None)
    assert st not in (INVALID, ALIAS, UNSUPPORTED)
    # ... but not inside the residual, which is written
    st = lib.rarn_fused_add_rms_norm_fp8(_fp8(A, H, mode=0, scale=C + 8), x, _rows(C, H, BF16),
                                         D, T, H, 1e-6, None)
    assert st == ALIAS
    # the codes span T rows of row_stride bytes: a scale right after it is fine
    st = lib.rarn_rms_norm_fp8(_fp8(A, 2 * H, mode=1, scale=A + 3 * 2 * H + H), x, D, T, H,
                               1e-6, None)
    assert st not in (INVALID, ALIAS, UNSUPPORTED)
    # the stream and cluster kernels have no 8-bit output
    for path in ("stream", "cluster"):
        rarn.set_path(path)
        try:
            assert lib.rarn_reduce_add_rms_norm_fp8(_fp8(A, H), x, T * H, 2, _rows(C, H, BF16), D,
                                                    T, H, 1e-6, None) == UNSUPPORTED
        finally:
            rarn.set_path("auto")
    assert lib.rarn_rms_norm_fp8(_fp8(None, H), _rows(None, H, BF16), None, 0, H, 1e-6,
                                 None) == OK


def test_plan_fp8():
    """The 8-bit output runs on the register row kernels for every shape."""
    cases = [("rms_norm", 30000, 512, 0, "warp", "pipe=1"),
             ("fused_add_rms_norm", 32768, 5120, 1, "rows.cta", "pipe=1"),
             ("fused_add_rms_norm", 16, 5120, 1, "rows.cta", "gamma_regs=1"),
             ("reduce_add_rms_norm", 8192, 8192, 8, "rows.cta", "vec16"),
             ("rms_norm", 4, 100000, 0, "rows.two_pass", "vec16")]
    for op, T, H, R, kind, flag in cases:
        p = rarn.plan_fp8(op, T, H, R, "bf16", num_sms=152)
        assert kind in p and flag in p, (op, T, H, p)
    assert "scalar" in rarn.plan_fp8("rms_norm", 64, 1000, 0, "bf16", vec_ok=False, num_sms=152)
    rarn.set_path("stream")
    try:
        assert rarn.plan_fp8("reduce_add_rms_norm", 8192, 8192, 8, "bf16",
                             num_sms=152).startswith("none")
    finally:
        rarn.set_path("auto")


def test_fp8_partials_argument_errors(lib):
    """Reduce over 8-bit partials: types, sizes, alignment and aliasing are
    checked before any CUDA call."""
    f = lib.rarn_reduce_add_rms_norm_fp8in
    T, H, R = 8, 1024, 4
    y, p, sc, r, g = A, B, C, D, D + (1 << 30)

    def call(y=y, p=p, R=R, fmt=0, sc=sc, r=r, g=g, T=T, H=H, eps=1e-6, dt=BF16):
        return f(y, p, R, fmt, sc, r, g, T, H, eps, dt, None)

    assert call(dt=7) == INVALID                       # unknown type
    assert call(fmt=2) == INVALID                      # unknown format
    assert call(R=0) == INVALID
    assert call(T=-1) == INVALID
    assert call(H=0) == INVALID
    assert call(eps=float("nan")) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(T=0, y=None, p=None, sc=None, r=None, g=None) == OK  # nothing to do
    assert call(sc=None) == INVALID
    assert call(p=None) == INVALID
    assert call(R=17) == UNSUPPORTED                   # at most 16 partials
    assert call(H=1020) == UNSUPPORTED                 # H a multiple of 8
    assert call(H=16392) == UNSUPPORTED                # at most 16384
    assert call(H=8200, dt=F32) == UNSUPPORTED         # binary32: at most 8192
    assert call(p=B + 4) == UNSUPPORTED                # codes 8-byte aligned
    assert call(r=D + 8) == UNSUPPORTED                # residual 16-byte aligned
    assert call(y=A + 8) == UNSUPPORTED
    assert call(sc=C + 2) == UNSUPPORTED
    assert call(y=D) == ALIAS                          # y over the residual
    assert call(r=B + 64) == ALIAS                     # residual over the codes
    assert call(y=C - 16) == ALIAS                     # y over the scales
    assert call(r=g - 16) == ALIAS                     # residual over gamma


def test_gemm_form_argument_errors(lib):
    """GEMM-producer form: types, shapes, workspace, alignment and aliasing
    are checked before any CUDA call."""
    T, H, K = 16, 1024, 256
    y, a, w, r = _rows(A, H, BF16), _rows(B, K, BF16), _rows(C, K, BF16), _rows(D, H, BF16)
    g = D + (1 << 30)
    ws, wsb = D + (2 << 30), 1 << 20
    f = lib.rarn_gemm_add_rms_norm

    def call(*args, wsp=ws, wsn=wsb):
        return f(*args, wsp, wsn, None)

    assert call(y, a, _rows(C, K, F16), r, g, T, H, K, 1e-6) == UNSUPPORTED  # mixed types
    assert call(y, a, w, r, g, T, H, K, -1.0) == INVALID                     # eps
    assert call(y, a, w, r, g, T, H, 0, 1e-6) == INVALID                     # K = 0
    assert call(y, _rows(B, K - 1, BF16), w, r, g, T, H, K, 1e-6) == INVALID  # row stride
    assert call(y, a, w, r, None, T, H, K, 1e-6) == INVALID                  # null gamma
    assert call(y, a, w, r, g, T, H, K, 1e-6, wsp=None) == INVALID           # no workspace
    need = lib.rarn_gemm_workspace_bytes(T, H)
    # partial sums [T][H / 128], one row-block counter, then (T <= 128) room for
    # split K: 9 x T x H binary32 partial products from a 256-byte boundary
    base = (T * (H // 128) + 1) * 4
    assert need == ((base // 4 + 63) // 64 * 64 + 9 * T * H) * 4
    # less than the split-K room only turns split K off; less than the base fails
    assert call(y, a, w, r, g, T, H, K, 1e-6, wsn=base - 4) == INVALID      # short workspace
    assert call(y, a, w, r, g, T, H, K, 1e-6, wsp=ws + 8) == INVALID         # not 16-byte aligned
    assert call(_rows(A, 300, BF16), a, _rows(C, K, BF16), _rows(D, 300, BF16), g, T, 300, K,
                1e-6) == UNSUPPORTED                                         # H = 300
    assert call(_rows(A, H, F32), _rows(B, K, F32), _rows(C, K, F32), _rows(D, H, F32), g, T, H,
                K, 1e-6) == UNSUPPORTED                                      # no f32 path
    assert call(y, _rows(B + 2, K, BF16), w, r, g, T, H, K, 1e-6) == UNSUPPORTED  # alignment
    assert call(y, _rows(B, K + 4, BF16), w, r, g, T, H, K, 1e-6) == UNSUPPORTED  # stride
    assert call(_rows(D, H, BF16), a, w, r, g, T, H, K, 1e-6) == ALIAS       # y == residual
    assert call(y, a, w, _rows(C + 64, H, BF16), g, T, H, K, 1e-6) == ALIAS  # residual over w
    assert call(y, a, w, r, g, T, H, K, 1e-6, wsp=A + 64) == ALIAS          # workspace over y
    assert call(_rows(None, H, BF16), _rows(None, K, BF16), _rows(None, K, BF16),
                _rows(None, H, BF16), None, 0, H, K, 1e-6, wsp=None) == OK  # T = 0


def test_plan_fp8in(tune):
    """Which kernel the reduce over 8-bit partials takes (pure host logic; a
    GB300's 152 SMs and 232448 bytes of opt-in shared memory per CTA)."""
    p = rarn.plan_fp8in(8192, 8192, 8)
    # the bench shape: 5 stages of 8 code chunks + a residual chunk of 4096
    # elements; the ncu capture of it reports 221.84 KB dynamic shared memory
    assert p == ("q8in.ring warps=16 ppt=1 chunk_elems=4096 stages=5 stage_bytes=40960 "
                 "smem=221840 grid=152 block=544"), p
    # four or three partials: the ring where the rows are long enough
    assert rarn.plan_fp8in(8192, 8192, 4).startswith("q8in.ring")
    assert rarn.plan_fp8in(16384, 4096, 4).startswith("q8in.ring")
    assert rarn.plan_fp8in(32768, 2048, 4) == "q8in.rows pack=16 vpt=1 block=128 grid=occupancy"
    assert rarn.plan_fp8in(8192, 8192, 3).startswith("q8in.ring")
    assert rarn.plan_fp8in(16384, 4096, 3) == "q8in.rows pack=16 vpt=1 block=256 grid=occupancy"
    assert rarn.plan_fp8in(32768, 4096, 2).startswith("q8in.rows")
    assert rarn.plan_fp8in(8 * 152 - 1, 8192, 4).startswith("q8in.rows")
    # rows shorter than 4096: the ring only from 8 partials
    assert rarn.plan_fp8in(32768, 2048, 6).startswith("q8in.rows")
    assert rarn.plan_fp8in(32768, 2048, 7).startswith("q8in.rows")
    assert rarn.plan_fp8in(32768, 2048, 8).startswith("q8in.ring")
    assert rarn.plan_fp8in(32768, 4096, 5).startswith("q8in.ring")
    assert rarn.plan_fp8in(8 * 152 - 1, 8192, 8).startswith("q8in.rows")  # < 8 rows per SM
    assert rarn.plan_fp8in(8 * 152, 8192, 8).startswith("q8in.ring")
    assert rarn.plan_fp8in(8192, 8200, 8) == "q8in.rows pack=8 vpt=8 block=160 grid=occupancy"
    assert rarn.plan_fp8in(8192, 8192, 8, codes_aligned16=False).startswith("q8in.rows")
    assert rarn.plan_fp8in(4096, 16384, 16).startswith("q8in.ring")
    assert rarn.plan_fp8in(8, 1020, 2).startswith("none")
    assert rarn.plan_fp8in(8, 16384, 2, "f32").startswith("none")
    tune(fp8in_pack16=0)
    assert rarn.plan_fp8in(64, 4096, 2) == "q8in.rows pack=8 vpt=2 block=256 grid=occupancy"
    tune(fp8in_ring=1)
    assert rarn.plan_fp8in(5, 512, 1).startswith("q8in.ring")
    assert rarn.plan_fp8in(5, 520, 1).startswith("q8in.rows")  # H not a multiple of 16
    tune(fp8in_ring=0)
    assert rarn.plan_fp8in(8192, 8192, 8).startswith("q8in.rows")


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_plan_fp8in_ring_fits(dt, tune):
    """The TMA-fed kernel forced on every partial count and a spread of row
    lengths: the ring always fits the opt-in shared memory with the row copy
    and control words, keeps at least 2 stages (4 with two units per
    thread), and every bulk copy is a whole number of 16-byte blocks."""
    tune(fp8in_ring=1)
    s = 4 if dt == "f32" else 2
    for R in range(1, 17):
        for H in (16, 1040, 4096, 8192, 8192 if dt == "f32" else 16384):
            p = rarn.plan_fp8in(1000, H, R, dt)
            assert p.startswith("q8in.ring"), (R, H, p)
            kv = {k: int(v) for k, v in (f.split("=") for f in p.split()[1:])}
            ppt, stages, sb, smem, chunk = (kv[k] for k in ("ppt", "stages", "stage_bytes",
                                                               "smem", "chunk_elems"))
            assert chunk == 512 * 8 * ppt
            assert stages >= (4 if ppt == 2 else 2) and smem <= 232448
            assert sb % 128 == 0 and sb >= R * chunk + chunk * s
            assert smem >= stages * sb + H * s
            last = H % chunk or chunk  # elements in a row's last chunk
            assert (last * 1) % 16 == 0 and (last * s) % 16 == 0


def test_plan_gemm(tune):
    """Columns per CTA from H; the K slab and ring depth fill one SM's shared
    memory; the workspace holds one float per row and column tile."""
    # persistent on SM pairs: 76 two-CTA clusters walk 256 tiles of 256 x 256,
    # each CTA staging 32 KB per K slab
    p = rarn.plan_gemm(4096, 4096, 4096)
    assert "cols_per_cta=256 col_tiles=16 bk=64 stages=3" in p and "grid=152" in p, p
    assert "kblocks=64 persistent=1 pair=1" in p, p
    p = rarn.plan_gemm(2100, 512, 512)     # 9 x 2 pair tiles: 18 clusters
    assert "grid=36 " in p and "pair=1" in p, p
    p = rarn.plan_gemm(1024, 4096, 4096)   # below 2048 rows, one round of 128 tiles: one SM per tile
    assert "persistent=1 pair=0" in p, p
    p = rarn.plan_gemm(1536, 4096, 4096)   # 192 one-SM tiles, more than a round: pairs
    assert "persistent=1 pair=1" in p, p
    p = rarn.plan_gemm(1536, 4096, 1024)   # ... but not for K below 2048
    assert "persistent=1 pair=0" in p, p
    # y in the epilogue where K >= 3072, or K >= 2048 with T >= 4096; else the
    # norm kernel after the GEMM
    for T, K, fused in ((4096, 4096, True), (4096, 3072, True), (4096, 2048, True),
                        (2048, 2048, False), (4096, 1024, False), (1536, 3072, True)):
        p = rarn.plan_gemm(T, 4096, K)
        assert ("norm in epilogue" in p) == fused and ("+ norm" in p) != fused, (T, K, p)
    tune(gemm_norm_in_epilogue=1)
    assert "norm in epilogue" in rarn.plan_gemm(4096, 4096, 1024)
    tune(gemm_norm_in_epilogue=0)
    assert "+ norm" in rarn.plan_gemm(4096, 4096, 4096)
    tune(gemm_norm_in_epilogue=-1)
    tune(gemm_pair=0)  # one CTA per SM walks 512 tiles of 128 x 256
    p = rarn.plan_gemm(4096, 4096, 4096)
    assert "cols_per_cta=256 col_tiles=16 bk=64 stages=4" in p and "grid=152" in p, p
    assert "kblocks=64 persistent=1 pair=0" in p, p
    tune(gemm_pair=-1)
    p = rarn.plan_gemm(200, 768, 960)      # two 128-row blocks, 15 K slabs: one SM per tile
    assert "cols_per_cta=256 col_tiles=3" in p and "persistent=1" in p and "grid=6" in p, p
    assert "pair=0" in p, p
    # tiles that leave half of the SMs idle: K split over the idle SMs, at
    # least 8 K slabs each, at most 9 splits, every row block
    p = rarn.plan_gemm(256, 4096, 4096)    # 2 x 16 tiles, 152 // 32 = 4 splits
    assert "splitk=4" in p and "grid=128" in p, p
    p = rarn.plan_gemm(512, 4096, 4096)    # 4 x 16 tiles: 2 splits
    assert "splitk=2" in p and "grid=128" in p, p
    p = rarn.plan_gemm(640, 4096, 4096)    # 5 x 16 tiles: more than half of the SMs
    assert "splitk" not in p and "persistent=1" in p, p
    p = rarn.plan_gemm(100, 768, 1000)
    assert "col_tiles=3" in p and "splitk=2" in p and "grid=6" in p, p
    p = rarn.plan_gemm(1, 4096, 4096)
    assert "col_tiles=16" in p and "splitk=8" in p and "grid=128" in p, p
    p = rarn.plan_gemm(16, 2048, 8192)
    assert "splitk=9" in p and "grid=72" in p, p
    tune(gemm_split_k=0)
    assert "persistent=1" in rarn.plan_gemm(1, 4096, 4096)
    tune(gemm_split_k=-1)
    p = rarn.plan_gemm(8, 16384, 64)   # beyond 32 tiles of 256: 512-column tiles
    assert "cols_per_cta=512 col_tiles=32 bk=32 stages=5" in p and "persistent=0" in p, p
    assert rarn.plan_gemm(8, 300, 64).startswith("none")
    assert rarn.plan_gemm(8, 16896, 64).startswith("none")   # 33 x 512: beyond 32 tiles
    assert rarn.plan_gemm(8, 4096, 64, "f32").startswith("none")
    # partial sums [T][H / 128], then one counter per 128-row block (16-byte
    # aligned); where split K can apply also room for min(9, 152 // tiles)
    # splits of T x H binary32 products from the next 256-byte boundary
    assert rarn.gemm_workspace_bytes(4096, 4096) == (4096 * 32 + 32) * 4
    assert rarn.gemm_workspace_bytes(1, 768) == (64 + 9 * 768) * 4
    base129 = (129 * 6 + 3) // 4 * 4 + 2
    assert rarn.gemm_workspace_bytes(129, 768) == ((base129 + 63) // 64 * 64 + 9 * 129 * 768) * 4
    base512 = 512 * 32 + 4
    assert rarn.gemm_workspace_bytes(512, 4096) == ((base512 + 63) // 64 * 64 + 2 * 512 * 4096) * 4
    assert rarn.gemm_workspace_bytes(640, 4096) == (640 * 32 + 5) * 4
    assert rarn.gemm_workspace_bytes(7, 300) == -1


# values each knob accepts besides -1 (include/rarn.h, rarn_tuning)
TUNING_OK = {
    "rows_per_thread": [1, 2, 4, 8, 16], "rows_grid": [1, 4096, 2 ** 31 - 1],
    "rows_pipeline": [0], "l2_rows": list(range(9)), "stream_packs": [1, 2, 4],
    "stream_groups": [1, 2], "gemm_cols": [256, 512], "gemm_slab": [32, 64],
    "gemm_ctas_per_sm": [1, 2], "gemm_persistent": [0, 1], "gemm_pair": [0, 1],
    "gemm_norm_in_epilogue": [0, 1], "gemm_tail_split": [0], "gemm_split_k": [0],
    "fp8in_ring": [0, 1], "fp8in_pack16": [0], "tp_prefetch": [0, 1],
}
TUNING_BAD = {
    "rows_per_thread": [0, 3, 32], "rows_grid": [0, 2 ** 31], "rows_pipeline": [1, -2],
    "l2_rows": [9, -2], "stream_packs": [0, 3, 8], "stream_groups": [0, 3],
    "gemm_cols": [128, 384], "gemm_slab": [16, 128], "gemm_ctas_per_sm": [0, 3],
    "gemm_persistent": [2], "gemm_pair": [2], "gemm_norm_in_epilogue": [2],
    "gemm_tail_split": [1], "gemm_split_k": [1, 9], "fp8in_ring": [2], "fp8in_pack16": [1],
    "tp_prefetch": [2, -2],
}


def test_tuning_knobs_validated(lib):
    """rarn_set_tuning accepts -1 and each knob's listed values, refuses
    everything else (status INVALID, the knob unchanged), and
    rarn_reset_tuning puts every knob back to -1."""
    assert set(TUNING_OK) == set(rarn.TUNING) == set(TUNING_BAD)
    assert sorted(rarn.TUNING.values()) == list(range(17))
    rarn.reset_tuning()
    try:
        for name, good in TUNING_OK.items():
            assert rarn.get_tuning(name) == -1
            for v in good:
                rarn.set_tuning(name, v)
                assert rarn.get_tuning(name) == v
            keep = good[0]
            rarn.set_tuning(name, keep)
            for v in TUNING_BAD[name]:
                with pytest.raises(rarn.RarnError) as e:
                    rarn.set_tuning(name, v)
                assert e.value.status == INVALID
                assert rarn.get_tuning(name) == keep, name
            rarn.set_tuning(name, -1)
        v = ctypes.c_int64(0)
        assert lib.rarn_set_tuning(17, 0) == INVALID   # no such knob
        assert lib.rarn_set_tuning(-1, 0) == INVALID
        assert lib.rarn_get_tuning(17, ctypes.byref(v)) == INVALID
        assert lib.rarn_get_tuning(0, None) == INVALID
        rarn.set_tuning("gemm_pair", 0)
        rarn.set_tuning("rows_grid", 7)
        rarn.reset_tuning()
        assert all(rarn.get_tuning(n) == -1 for n in rarn.TUNING)
    finally:
        rarn.reset_tuning()


def test_tuning_steers_the_planners(tune):
    """Knobs reach the row, stream, GEMM and 8-bit-partials planners (pure
    host logic: the plan queries with a GB300's SM count)."""
    base = rarn.plan("fused_add_rms_norm", 4096, 4096, 1, "bf16", num_sms=152)
    assert "pipe=1" in base and "per_thread=2" in base, base
    tune(rows_pipeline=0, rows_per_thread=4, rows_grid=300)
    p = rarn.plan("fused_add_rms_norm", 4096, 4096, 1, "bf16", num_sms=152)
    assert "pipe=0" in p and "per_thread=4" in p and "grid=300" in p, p
    tune(stream_packs=1)
    p = rarn.plan("reduce_add_rms_norm", 8192, 8192, 8, "bf16", num_sms=152)
    assert p.startswith("stream") and "chunk=4096" in p, p
    tune(gemm_cols=512, gemm_slab=64, gemm_ctas_per_sm=1)
    p = rarn.plan_gemm(4096, 4096, 4096)
    assert "cols_per_cta=512" in p and "bk=64" in p and "persistent=0" in p, p
    tune(fp8in_ring=0)
    assert rarn.plan_fp8in(8192, 8192, 8).startswith("q8in.rows")
    rarn.reset_tuning()
    assert rarn.plan("fused_add_rms_norm", 4096, 4096, 1, "bf16", num_sms=152) == base


def test_plan_gemm_takes_the_sm_count():
    """The GEMM planner sizes its persistent grid and split K from the SM
    count it is given (the compute call passes the device's)."""
    p = rarn.plan_gemm(4096, 4096, 4096, num_sms=132)
    assert "grid=132" in p and "pair=1" in p, p
    p = rarn.plan_gemm(1, 4096, 4096, num_sms=64)   # 64 SMs / 16 column tiles: 4 splits
    assert "splitk=4" in p and "grid=64" in p, p
    assert "splitk=8" in rarn.plan_gemm(1, 4096, 4096, num_sms=152)


def test_noalloc_rows_match_the_header(lib):
    """The rows one launch sequence of the allocation-free GEMM entry point
    covers: floor(floor((2^20 - 16) / (H / 128 + 1)) / 128) * 128, and the
    figures the header quotes for H = 8192 and 16384."""
    with open(HEADER) as f:
        text = f.read()
    assert "16128 rows at H = 8192, 8064 at H = 16384" in text
    assert rarn.gemm_noalloc_rows(8192) == 16128
    assert rarn.gemm_noalloc_rows(16384) == 8064
    for H in (256, 512, 768, 1024, 4096, 5120, 8192, 12288, 16384):
        assert rarn.gemm_noalloc_rows(H) == (2 ** 20 - 16) // (H // 128 + 1) // 128 * 128, H
        rows = rarn.gemm_noalloc_rows(H)
        # partial sums [rows][H / 128], then one counter per 128-row block
        assert (rows * (H // 128) + 3) // 4 * 4 + rows // 128 <= 2 ** 20
    assert rarn.gemm_noalloc_rows(300) == -1
    assert rarn.gemm_noalloc_rows(16896) == -1


def test_noalloc_checks_the_whole_call_first(lib):
    """The allocation-free GEMM entry point validates all T rows before it
    launches any chunk: outputs of one chunk overlapping another chunk's
    inputs are refused (RARN_ERR_ALIAS), as the workspace form refuses them,
    and so are argument errors that only a later chunk would meet.  No call
    here reaches the GPU."""
    H, K = 8192, 64
    chunk = rarn.gemm_noalloc_rows(H)
    T = 2 * chunk
    f = lib.rarn_gemm_add_rms_norm_noalloc
    g = D + (1 << 36)
    a, w = _rows(B, K, BF16), _rows(C, K, BF16)
    r = _rows(A, H, BF16)
    # y starts where the second chunk's residual rows start: chunk 0 would
    # overwrite rows that chunk 1 then reads
    y = _rows(A + chunk * H * 2, H, BF16)
    assert f(y, a, w, r, g, T, H, K, 1e-6, None) == ALIAS
    ws = D + (1 << 38)
    assert lib.rarn_gemm_add_rms_norm(y, a, w, r, g, T, H, K, 1e-6, ws, 1 << 30, None) == ALIAS
    # A's last chunk over y's first rows
    y2 = _rows(D, H, BF16)
    a2 = _rows(D - (T - 1) * K * 2, K, BF16)
    assert f(y2, a2, w, r, g, T, H, K, 1e-6, None) == ALIAS
    # the other argument errors of the workspace form, before any CUDA call
    assert f(y2, a, w, r, g, T, H, K, -1.0, None) == INVALID
    assert f(y2, a, _rows(C, K, F16), r, g, T, H, K, 1e-6, None) == UNSUPPORTED
    assert f(y2, a, w, r, g, T, 300, K, 1e-6, None) == UNSUPPORTED
    assert f(y2, _rows(B + 2, K, BF16), w, r, g, T, H, K, 1e-6, None) == UNSUPPORTED
    assert f(_rows(None, H, BF16), a, w, r, g, 0, H, K, 1e-6, None) == OK  # T = 0


def test_launch_floor_argument_errors(lib):
    """The launch-floor measurement aid rejects bad shapes and row arguments
    before any CUDA call."""
    f = lib.rarn_launch_floor
    assert f(None, 0, 0, 256, None) == INVALID
    assert f(None, 0, 4, 0, None) == INVALID
    assert f(None, 0, 4, 1025, None) == INVALID
    assert f(A, 0, 4, 256, None) == INVALID           # row of 0 bytes
    assert f(A, 24, 4, 256, None) == INVALID          # not a multiple of 16
    assert f(A, 2 ** 20 + 16, 4, 256, None) == INVALID
    assert f(A + 8, 16, 4, 256, None) == INVALID      # not 16-byte aligned
