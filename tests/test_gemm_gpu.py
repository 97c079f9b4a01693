"""GPU parity of the GEMM producer with the fused residual-add RMSNorm
epilogue (tcgen05 tensor cores and TMA; the column tiles' partial sums of
squares meet in a workspace read by the norm kernel) against the CPU oracle.

Bar.  The kernel accumulates P = A W^T in binary32 on the tensor cores; the
oracle has P exactly.  So the updated residual h must be a correct rounding
of some value within the accumulation error of P + r: RN(P + r - B) <= h <=
RN(P + r + B), with B = (ceil(K / 16) + 8) * 2^-23 * sum_k |A_tk W_ik| plus
one binary32 rounding of the sum -- a binary32 accumulation in 16-element
chunks.  Away from cancellation that is h = RN(P + r) or its neighbour at a
near-tie.  y must be within 2 units in the last place of the oracle's y plus
the residual's own distance at that element (y is computed from h)."""
import math

import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from residual_add_rmsnorm_gb300 import workloads as W

from gpu_util import to_device, to_host
from pins import lib_decode, ulp_dist

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset():
    yield
    rarn.set_pdl(True)


def gemm_inputs(T, H, K, dt, seed):
    """A ~ N(0, 1), W ~ N(0, 1 / K) (so P ~ N(0, 1)), residual ~ N(0, 1),
    gamma ~ U(0.5, 1.5), as storage bits."""
    rng = np.random.default_rng(seed)
    A = W.to_storage(rng.standard_normal((T, K)).astype(np.float32), dt)
    Wt = W.to_storage((rng.standard_normal((H, K)) / math.sqrt(K)).astype(np.float32), dt)
    R = W.to_storage(rng.standard_normal((T, H)).astype(np.float32), dt)
    G = W.to_storage(rng.uniform(0.5, 1.5, H).astype(np.float32), dt)
    return A, Wt, R, G


def ulp_of(v, dt):
    """Unit in the last place of the storage-format values v (binary64)."""
    p, emin = {"bf16": (8, -126), "f16": (11, -14), "f32": (24, -126)}[dt]
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(np.where(a > 0, e, emin), emin)
    return np.exp2(e - (p - 1))


def check_gemm(ref, K, y, res, dt, what, rows=None):
    """ref: oracle Result (residual, y, p64, abs64) for the rows checked."""
    T, H = ref.p64.shape
    r_in = ref.r_in
    exact = ref.p64 + r_in
    B = (math.ceil(K / 16) + 8) * 2.0 ** -23 * ref.abs64
    B = B + 2.0 ** -24 * (np.abs(exact) + B)
    O = oracle.default()
    lo = lib_decode(O.round_to(exact - B, dt), dt)
    hi = lib_decode(O.round_to(exact + B, dt), dt)
    h = lib_decode(res, dt).reshape(T, H)
    outside = (h < lo) | (h > hi)
    assert not outside.any(), (f"{what}: {int(outside.sum())} residual elements outside the "
                               f"accumulation bound, e.g. {np.argwhere(outside)[:3].tolist()}")
    # y = RN((h inv) gamma): the GPU's h may differ from the oracle's by the
    # amount allowed above; that difference scales by inv |gamma| into y, on
    # top of two units in the last place of y (two roundings, inv's binary32
    # evaluation)
    h_o = lib_decode(ref.residual, dt).reshape(T, H)
    y_o = lib_decode(ref.y, dt).reshape(T, H)
    y_g = lib_decode(y, dt).reshape(T, H)
    allow = 2 * ulp_of(y_o, dt) + np.abs(h - h_o) * ref.inv[:, None] * np.abs(ref.gamma) * 1.01
    over = np.abs(y_g - y_o) > allow
    assert not over.any(), (f"{what}: {int(over.sum())} y elements beyond 2 ulps plus the "
                            f"residual's difference, e.g. {np.argwhere(over)[:3].tolist()}")


def run_case(T, H, K, dt="bf16", seed=0, lda=None, ldw=None, ldr=None, ldy=None, eps=1e-6,
             sample_rows=None):
    import torch
    lda, ldw, ldr, ldy = lda or K, ldw or K, ldr or H, ldy or H
    A, Wt, R, G = gemm_inputs(T, H, K, dt, seed)

    def strided(bits, rows, cols, ld):
        full = torch.zeros(rows, ld, dtype=to_device(bits[:1], dt).dtype, device="cuda")
        full[:, :cols] = to_device(bits, dt)
        return full, full[:, :cols]

    _, a = strided(A, T, K, lda)
    _, w = strided(Wt, H, K, ldw)
    rfull, r = strided(R, T, H, ldr)
    yfull, y = strided(np.zeros((T, H), R.dtype), T, H, ldy)
    g = to_device(G, dt)
    plan = rarn.plan_gemm(T, H, K, dt)
    rarn.gemm_add_rms_norm(a, w, r, g, eps, out=y)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    rows = np.arange(T) if sample_rows is None else sample_rows
    As = np.ascontiguousarray(A[rows])
    Rs = np.ascontiguousarray(R[rows]).reshape(-1).copy()
    ref = oracle.gemm_add_rms_norm(dt, As.reshape(-1), Wt.reshape(-1), Rs, G, eps, len(rows), H,
                                   K, want_p64=True)
    ref.residual = ref.residual.reshape(len(rows), H)
    ref.y = ref.y.reshape(len(rows), H)
    ref.r_in = lib_decode(R[rows], dt)
    ref.gamma = lib_decode(G, dt)
    res_h = to_host(r.contiguous(), dt)[rows]
    y_h = to_host(y.contiguous(), dt)[rows]
    check_gemm(ref, K, y_h, res_h, dt, f"gemm {dt} T{T} H{H} K{K} ({plan})")
    # padding of the strided outputs untouched
    if ldr > H:
        assert torch.all(rfull[:, H:] == 0)
    if ldy > H:
        assert torch.all(yfull[:, H:] == 0)
    return plan


@pytest.mark.parametrize("T,H,K", [
    (128, 512, 64),      # 2 column tiles of 256, one K slab
    (200, 1024, 200),    # ragged rows and K, the 2-stage ring wraps
    (256, 4096, 1024),   # 16 column tiles
    (300, 768, 512),     # 3 column tiles
    (1, 2048, 4096),     # one row (decode), long K
    (77, 8192, 256),     # 32 column tiles of 256
    (130, 5120, 320),    # 20 column tiles
    (40, 16384, 128),    # 32 column tiles of 512 (one CTA per SM, 64-byte K slabs)
])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_gemm_parity(T, H, K, dt):
    plan = run_case(T, H, K, dt, seed=T + H + K)
    assert plan.startswith("gemm.tcgen05"), plan
    # split K where the 128 x 256 tiles leave at least half of the 152 SMs idle
    tiles = -(-T // 128) * (H // 256)
    splitk = H <= 8192 and min(9, 152 // tiles, -(-K // 64) // 8) >= 2
    assert ("splitk=" in plan) == splitk, plan
    assert ("persistent=1" in plan) == (H <= 8192 and K >= 512 and not splitk), plan
    pair = H <= 8192 and K >= 512 and not splitk and (
        T >= 2048 or (K >= 2048 and -(-T // 128) * (H // 256) > 152))
    assert ("pair=1" in plan) == pair, plan


@pytest.mark.parametrize("T,H,K,fused", [
    (1280, 4096, 2048, False),   # pairs below 2048 rows (160 one-SM tiles), y by the norm kernel
    (1536, 5120, 3072, True),    # ... with y in the epilogue (K >= 3072)
])
def test_gemm_mid_rows_on_pairs(T, H, K, fused):
    """The planner's SM pairs where one SM per 128-row tile would need more
    than one round of the SMs, and its choice of where y is formed; sampled
    rows against the oracle."""
    plan = run_case(T, H, K, "bf16", seed=T + K, sample_rows=np.arange(0, T, 13))
    assert "pair=1" in plan and ("norm in epilogue" in plan) == fused, plan


@pytest.mark.parametrize("ns,bk,ctas", [(256, 32, 2), (256, 64, 2), (256, 64, 1), (512, 32, 1),
                                        (512, 64, 1)])
def test_gemm_tilings(ns, bk, ctas, tune):
    """The non-persistent kernel in every tiling the planner can choose
    (tuning knobs): 256 / 512 columns per CTA, 64-byte and 128-byte
    swizzled K slabs, one or two CTAs per SM.  (The default, persistent kernel
    runs in every other test.)"""
    tune(gemm_cols=ns, gemm_slab=bk, gemm_ctas_per_sm=ctas)
    for T, H, K in ((256, 1024, 448), (64, 512, 1000), (300, 2048, 2048)):
        plan = run_case(T, H, K, "bf16", seed=K)
        assert f"cols_per_cta={ns}" in plan and f"bk={bk}" in plan, plan
        assert "persistent=0" in plan, plan


@pytest.mark.parametrize("pair", [0, 1])
def test_gemm_persistent_one_sm_and_sm_pairs(pair, tune):
    """The persistent kernel forced onto one SM per 128 x 256 tile and onto
    SM pairs (two-CTA clusters, cta_group::2 MMAs on 256 x 256 tiles, each CTA
    staging half of the W slab): one row, ragged rows and K, a single K slab,
    3 to 32 column tiles, and more tiles than pairs so that both accumulators
    are reused."""
    tune(gemm_persistent=1, gemm_pair=pair)
    for T, H, K, dt in ((1, 1024, 512, "bf16"), (200, 768, 520, "bf16"),
                        (300, 2048, 1024, "f16"), (700, 1536, 64, "bf16"),
                        (520, 8192, 192, "bf16"), (2500, 4096, 96, "bf16")):
        plan = run_case(T, H, K, dt, seed=T + K + 7)
        assert "persistent=1" in plan and f"pair={pair}" in plan, plan
    # residual rows that do not all start on a 32-byte boundary (row stride
    # 1032): the epilogue's 16-byte form
    plan = run_case(300, 1024, 512, "bf16", seed=3, ldr=1032, ldy=1040)
    assert "persistent=1" in plan and f"pair={pair}" in plan, plan


@pytest.mark.parametrize("pair", [0, 1])
def test_gemm_norm_in_epilogue_matches_norm_kernel(pair, tune):
    """y written by the persistent kernel's epilogue (each tile waits on its
    128-row block's counter) and by the separate norm kernel: bit-identical,
    on shapes with more tiles than CTAs or pairs, so that row blocks straddle
    two rounds of tiles, and with 32 column tiles per row.  At 4096 rows on
    pairs some pairs defer the y of two items in a row (a row block
    straddling rounds 0 and 1, another rounds 1 and 2), the case where the
    staged gamma must not be overwritten while a deferred y still reads it."""
    import torch
    tune(gemm_pair=pair, gemm_split_k=0)  # the persistent kernels, not split K
    for T, H, K in ((2500, 4096, 512), (1000, 8192, 576), (129, 2048, 1024), (4096, 4096, 512)):
        gen = torch.Generator(device="cuda").manual_seed(T + H + K)
        a = torch.randn(T, K, device="cuda", generator=gen).to(torch.bfloat16)
        w = (torch.randn(H, K, device="cuda", generator=gen) / K ** 0.5).to(torch.bfloat16)
        r0 = torch.randn(T, H, device="cuda", generator=gen).to(torch.bfloat16)
        g = (torch.rand(H, device="cuda", generator=gen) + 0.5).to(torch.bfloat16)
        outs = {}
        for fuse in (1, 0):
            tune(gemm_norm_in_epilogue=fuse)
            plan = rarn.plan_gemm(T, H, K)
            assert ("norm in epilogue" in plan) == (fuse == 1), plan
            r = r0.clone()
            y = rarn.gemm_add_rms_norm(a, w, r, g, 1e-6)
            torch.cuda.synchronize()
            assert rarn.watchdog(clear=True) == 0
            outs[fuse] = (y, r)
        assert torch.equal(outs[1][0], outs[0][0]), f"y differs at T{T} H{H} K{K}"
        assert torch.equal(outs[1][1], outs[0][1]), f"residual differs at T{T} H{H} K{K}"


def test_gemm_pair_tail_halves(tune):
    """The pair kernel's last partial round as 128-column halves (N = 128
    MMAs; a round then fills up to twice as many SM pairs) against whole
    tiles: bit-identical (the same K order per element, the same 128-column
    partial sums); sampled rows against the oracle."""
    import torch
    tune(gemm_pair=1)
    plan = run_case(1536, 4096, 512, "bf16", seed=9, sample_rows=np.arange(1280, 1536, 4))
    assert "tail=halves" in plan, plan
    for T, H, K in ((1536, 4096, 512), (2560, 2048, 576)):
        gen = torch.Generator(device="cuda").manual_seed(T + K)
        a = torch.randn(T, K, device="cuda", generator=gen).to(torch.bfloat16)
        w = (torch.randn(H, K, device="cuda", generator=gen) / K ** 0.5).to(torch.bfloat16)
        r0 = torch.randn(T, H, device="cuda", generator=gen).to(torch.bfloat16)
        g = (torch.rand(H, device="cuda", generator=gen) + 0.5).to(torch.bfloat16)
        outs = {}
        for split in (-1, 0):
            tune(gemm_tail_split=split)
            plan = rarn.plan_gemm(T, H, K)
            assert ("tail=halves" in plan) == (split == -1) and "pair=1" in plan, plan
            r = r0.clone()
            y = rarn.gemm_add_rms_norm(a, w, r, g, 1e-6)
            torch.cuda.synchronize()
            assert rarn.watchdog(clear=True) == 0
            outs[split] = (y, r)
        dy = (outs[-1][0] != outs[0][0])
        dr = (outs[-1][1] != outs[0][1])
        rows_y = torch.nonzero(dy.any(1)).flatten().tolist()
        cols_y = torch.nonzero(dy.any(0)).flatten().tolist()
        assert not dy.any() and not dr.any(), (
            f"T{T} H{H} K{K}: {int(dy.sum())} y / {int(dr.sum())} residual elements differ; "
            f"rows {rows_y[:4]}..{rows_y[-4:]} ({len(rows_y)}), cols {cols_y[:4]}..{cols_y[-4:]} "
            f"({len(cols_y)})")


@pytest.mark.parametrize("T,H,K,dt", [
    (1, 4096, 4096, "bf16"),    # decode: 16 column tiles x 8 splits
    (16, 768, 1000, "bf16"),    # ragged K, 2 splits
    (100, 2048, 4096, "f16"),   # 8 splits of 8 slabs
    (128, 8192, 2048, "bf16"),  # 32 column tiles x 4 splits
    (5, 2048, 8192, "bf16"),    # 9 splits (the most), 15 slabs each, the last 8
    (256, 4096, 4096, "bf16"),  # 2 row blocks x 16 column tiles x 4 splits
    (300, 2048, 1024, "f16"),   # 3 row blocks (the last ragged) x 8 tiles x 2 splits
    (512, 4096, 2048, "bf16"),  # 4 row blocks x 16 tiles x 2 splits
    (3, 4096, 2048, "f16"),     # the split sum and norm on a cluster of 8 CTAs per row
    (12, 8192, 2048, "bf16"),   # ... for up to 16 rows of 8192 columns
])
def test_gemm_splitk(T, H, K, dt):
    """Split K where the 128 x 256 tiles leave half of the SMs idle: M x C x
    splits CTAs (row block, column tile, K range) write binary32 partial
    products, a CTA per row (a cluster of 8 for very few rows) adds them in
    split order, adds the residual (one rounding) and normalises; against the
    oracle with the accumulation bound (at most 8 extra binary32 additions per
    element)."""
    plan = run_case(T, H, K, dt, seed=T * 7 + K)
    assert "splitk=" in plan, plan


def test_gemm_splitk_off_matches_oracle_too(tune):
    """The same single-row-block shapes without split K (the persistent
    kernel): both stay within the bound; split K is a different, equally
    valid binary32 summation order."""
    tune(gemm_split_k=0)
    for T, H, K in ((1, 4096, 4096), (100, 2048, 4096)):
        plan = run_case(T, H, K, "bf16", seed=T * 7 + K)
        assert "splitk=" not in plan and "persistent=1" in plan, plan


def test_gemm_strides():
    """Row strides for every matrix; padding of the outputs untouched."""
    run_case(150, 1024, 136, "bf16", seed=5, lda=200, ldw=144, ldr=1096, ldy=1032)


@pytest.mark.parametrize("pdl", [True, False])
def test_gemm_chained_with_norm_kernels(pdl):
    """A chain on one stream: GEMM + norm, the fused norm kernel on its
    output, the GEMM again -- the residual carries over; PDL on and off."""
    import torch
    rarn.set_pdl(pdl)
    T, H, K = 512, 2048, 512
    A, Wt, R, G = gemm_inputs(T, H, K, "bf16", 11)
    a, w, r, g = (to_device(A, "bf16"), to_device(Wt, "bf16"), to_device(R, "bf16"),
                  to_device(G, "bf16"))
    y = rarn.gemm_add_rms_norm(a, w, r, g, 1e-6)
    rarn.fused_add_rms_norm(y, r, g, 1e-6)   # residual += y
    y2 = rarn.gemm_add_rms_norm(a, w, r, g, 1e-6)
    torch.cuda.synchronize()
    # replay on the host side with the oracle, step by step, from the GPU's
    # inputs only (no GPU value feeds the oracle)
    res = R.reshape(-1).copy()
    o1 = oracle.gemm_add_rms_norm("bf16", A.reshape(-1), Wt.reshape(-1), res, G, 1e-6, T, H, K)
    o2 = oracle.fused_add_rms_norm(o1.y.reshape(T, H), o1.residual.reshape(T, H), G, 1e-6,
                                   "bf16")
    res2 = o2.residual.reshape(-1).copy()
    o3 = oracle.gemm_add_rms_norm("bf16", A.reshape(-1), Wt.reshape(-1), res2, G, 1e-6, T, H, K)
    # the chain amplifies near-tie roundings only slightly: compare in ulps
    d_r = ulp_dist(to_host(r, "bf16").reshape(-1), o3.residual, "bf16")
    d_y = ulp_dist(to_host(y2, "bf16").reshape(-1), o3.y, "bf16")
    assert np.percentile(d_r, 99.9) <= 1 and np.percentile(d_y, 99.9) <= 2
    assert np.mean(d_r == 0) > 0.999 and np.mean(d_y <= 1) > 0.999


def test_gemm_full_size_sampled():
    """The benchmark workload (T = K = H = 4096, bf16, the benchmark's input
    recipe) in its launch configuration; the oracle checks 64 sampled rows."""
    import torch
    gw = W.GEMM_CONFIGS[0]
    d = W.generate_gemm(gw)
    a, w, r, g = (to_device(d[k], gw.dtype) for k in ("a", "w", "residual", "gamma"))
    y = rarn.gemm_add_rms_norm(a, w, r, g, gw.eps)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    rows = np.linspace(0, gw.T - 1, 64).astype(int)
    res_in = np.ascontiguousarray(d["residual"][rows])
    ref = oracle.gemm_add_rms_norm(gw.dtype, np.ascontiguousarray(d["a"][rows]).reshape(-1),
                                   d["w"].reshape(-1), res_in.reshape(-1).copy(), d["gamma"],
                                   gw.eps, len(rows), gw.H, gw.K, want_p64=True)
    ref.residual = ref.residual.reshape(len(rows), gw.H)
    ref.y = ref.y.reshape(len(rows), gw.H)
    ref.r_in = lib_decode(res_in, gw.dtype)
    ref.gamma = lib_decode(d["gamma"], gw.dtype)
    check_gemm(ref, gw.K, to_host(y, gw.dtype)[rows], to_host(r, gw.dtype)[rows], gw.dtype,
               gw.name)
    assert "col_tiles=16" in rarn.plan_gemm(gw.T, gw.H, gw.K, gw.dtype)


def test_gemm_rejects():
    import torch
    a = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(300, 64, dtype=torch.bfloat16, device="cuda")
    r = torch.zeros(8, 300, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(300, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rarn.RarnError):  # H = 300: no column tiling
        rarn.gemm_add_rms_norm(a, w, r, g, 1e-6)
    a32 = torch.zeros(8, 64, dtype=torch.float32, device="cuda")
    w32 = torch.zeros(512, 64, dtype=torch.float32, device="cuda")
    r32 = torch.zeros(8, 512, dtype=torch.float32, device="cuda")
    g32 = torch.zeros(512, dtype=torch.float32, device="cuda")
    with pytest.raises(rarn.RarnError):  # f32: no tensor path
        rarn.gemm_add_rms_norm(a32, w32, r32, g32, 1e-6)
