"""The tensor-parallel form (reduce-scatter, residual add + RMSNorm,
all-gather) on one GPU, against the oracle.

The N ranks are N separate buffers on this device: every rank's part in one
launch (cooperative when the ranks meet in their signal-pad barriers), or the
ranks' launches one after another with no barrier, or two processes sharing
their buffers through CUDA IPC with host barriers between the steps.  No
launch here waits on another launch.  The bar: every rank's buffer holds y
for all T rows (2 ulps / 1e-5 relative, as everywhere), each rank's residual
rows bit-exact."""
import os
import socket
import sys

import numpy as np
import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn
from gpu_util import assert_bits_equal, assert_y_close, to_device, to_host
from residual_add_rmsnorm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EPS = 1e-6


def _inputs(N, T, H, dt, seed):
    w = W.workload("reduce_add_rms_norm", dt, T, H, R=N, eps=EPS, seed=seed,
                   partial_std=1.0 / np.sqrt(N))
    return W.generate(w)


def _device_group(d, N, T, H, dt, signals):
    import torch
    bufs = [to_device(d["partials"][q], dt) for q in range(N)]
    res = []
    for q in range(N):
        r0, r1 = rarn.tp_rows(T, N, q)
        res.append(to_device(np.ascontiguousarray(d["residual"][r0:r1]), dt))
    g = to_device(d["gamma"], dt)
    pads = ([torch.zeros(rarn.TP_SIGNAL_BYTES // 4, dtype=torch.int32, device="cuda")
             for _ in range(N)] if signals else None)
    return bufs, res, g, pads


def _check(bufs, res, ref, N, T, dt, what):
    for q in range(N):
        assert_y_close(to_host(bufs[q], dt), ref.ys[q], dt, f"{what} y in rank {q}'s buffer")
        r0, r1 = rarn.tp_rows(T, N, q)
        assert_bits_equal(to_host(res[q], dt), ref.residual[r0:r1], f"{what} rank {q} residual")


CASES = [  # N, T, H, dtype
    (1, 33, 1024, "bf16"),
    (2, 100, 4096, "bf16"),
    (3, 7, 2048, "f16"),
    (4, 1000, 8192, "bf16"),
    (8, 257, 5120, "bf16"),     # 640 packs: two per thread
    (8, 3, 16384, "bf16"),      # fewer rows than ranks; 2048 packs: four per thread
    (5, 64, 768, "f32"),
    (4, 300, 8192, "f32"),      # 2048 packs of binary32
    (8, 1, 512, "f16"),
]


@pytest.mark.parametrize("signals", [False, True])
@pytest.mark.parametrize("N,T,H,dt", CASES)
def test_tp_world_matches_oracle(N, T, H, dt, signals):
    """Every rank's part in one launch; with signal pads the ranks' CTAs
    meet in the entry and exit barriers (a cooperative launch)."""
    import torch
    d = _inputs(N, T, H, dt, seed=N * 1000 + T)
    ref = oracle.tp_reduce_add_rms_norm([d["partials"][q] for q in range(N)], d["residual"],
                                        d["gamma"], EPS, dt)
    bufs, res, g, pads = _device_group(d, N, T, H, dt, signals)
    rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref, N, T, dt, f"N{N} T{T} H{H} {dt}")
    if pads is not None:  # every flag consumed: the pads are ready for the next call
        for p in pads:
            assert int(p.abs().sum()) == 0


@pytest.mark.parametrize("prefetch", [0, 1])
@pytest.mark.parametrize("N,T,H,dt,signals", [
    (2, 2048, 8192, "bf16", True),    # 14 rows per CTA
    (2, 2047, 5120, "bf16", False),   # ragged: rank 0 owns 1023 rows, rank 1 1024
    (4, 4000, 4096, "f32", True),
    (1, 1500, 2048, "f16", False),
    (8, 3000, 8192, "bf16", True),
])
def test_tp_next_row_prefetch(N, T, H, dt, signals, prefetch, tune):
    """Each CTA works through many rows with the next-row L2 prefetch forced
    off and on: the same results as the oracle either way (the prefetch only
    moves data into L2 earlier)."""
    import torch
    tune(tp_prefetch=prefetch)
    plan = rarn.plan_tp(T, H, N, dt, True, 0, 0)
    assert f"prefetch={prefetch}" in plan, plan
    d = _inputs(N, T, H, dt, seed=31 + N + T)
    ref = oracle.tp_reduce_add_rms_norm([d["partials"][q] for q in range(N)], d["residual"],
                                        d["gamma"], EPS, dt)
    bufs, res, g, pads = _device_group(d, N, T, H, dt, signals)
    rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref, N, T, dt, f"N{N} T{T} H{H} {dt} prefetch={prefetch}")


def test_tp_ranks_in_turn_with_prefetch(tune):
    """The per-rank entry point with the prefetch forced on: each rank's
    launch prefetches its own residual and every buffer (all of this
    device's memory here)."""
    import torch
    tune(tp_prefetch=1)
    N, T, H, dt = 2, 3000, 4096, "bf16"
    d = _inputs(N, T, H, dt, seed=77)
    ref = oracle.tp_reduce_add_rms_norm([d["partials"][q] for q in range(N)], d["residual"],
                                        d["gamma"], EPS, dt)
    bufs, res, g, _ = _device_group(d, N, T, H, dt, False)
    for r in range(N):
        rarn.tp_reduce_add_rms_norm(bufs, r, res[r], g, EPS, T)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref, N, T, dt, "in turn, prefetch on")


@pytest.mark.parametrize("N,T,H,dt", [(2, 100, 4096, "bf16"), (4, 1000, 8192, "bf16"),
                                      (3, 7, 2048, "f16"), (5, 64, 768, "f32")])
def test_tp_ranks_one_after_another(N, T, H, dt):
    """The per-rank entry point, ranks launched in turn on one stream with no
    signal pads (the caller orders the ranks): rank r reads only its own rows
    of every buffer and writes only those rows, so the sequence gives the
    same result as N GPUs running at once."""
    import torch
    d = _inputs(N, T, H, dt, seed=7 + N)
    ref = oracle.tp_reduce_add_rms_norm([d["partials"][q] for q in range(N)], d["residual"],
                                        d["gamma"], EPS, dt)
    bufs, res, g, _ = _device_group(d, N, T, H, dt, False)
    for r in range(N):
        rarn.tp_reduce_add_rms_norm(bufs, r, res[r], g, EPS, T)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref, N, T, dt, f"N{N} T{T} H{H} {dt} in turn")


def test_tp_per_rank_barrier_on_one_gpu_is_refused():
    """Per-rank calls that meet in signal-pad barriers need their ranks on
    different GPUs; with every buffer on this one the call returns
    UNSUPPORTED before launching, and the buffers are untouched."""
    import torch
    N, T, H, dt = 2, 64, 1024, "bf16"
    d = _inputs(N, T, H, dt, seed=21)
    bufs, res, g, pads = _device_group(d, N, T, H, dt, True)
    with pytest.raises(rarn.RarnError) as e:
        rarn.tp_reduce_add_rms_norm(bufs, 0, res[0], g, EPS, T, signals=pads)
    assert e.value.status == 2
    torch.cuda.synchronize()
    for q in range(N):
        assert_bits_equal(to_host(bufs[q], dt), d["partials"][q], f"rank {q}'s buffer")
        assert int(pads[q].abs().sum()) == 0


@pytest.mark.parametrize("signals", [False, True])
@pytest.mark.parametrize("pdl", [True, False])
def test_tp_two_steps(pdl, signals):
    """Two layers in a row on one stream: the second step's partials are
    written over the first step's y, and its residual is the one the first
    step stored; replayed with the oracle."""
    import torch
    N, T, H, dt = 4, 200, 4096, "bf16"
    d1 = _inputs(N, T, H, dt, seed=1)
    d2 = _inputs(N, T, H, dt, seed=2)
    ref1 = oracle.tp_reduce_add_rms_norm([d1["partials"][q] for q in range(N)], d1["residual"],
                                         d1["gamma"], EPS, dt)
    ref2 = oracle.tp_reduce_add_rms_norm([d2["partials"][q] for q in range(N)], ref1.residual,
                                         d1["gamma"], EPS, dt)
    rarn.set_pdl(pdl)
    try:
        bufs, res, g, pads = _device_group(d1, N, T, H, dt, signals)
        nxt = [to_device(d2["partials"][q], dt) for q in range(N)]
        rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
        for q in range(N):
            bufs[q].copy_(nxt[q])
        rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
        torch.cuda.synchronize()
    finally:
        rarn.set_pdl(True)
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref2, N, T, dt, f"two steps pdl={pdl}")


@pytest.mark.parametrize("stall_rank", [0, 3])
def test_tp_barrier_wait_runs_out_and_is_reported(stall_rank):
    """CTA 0 of one rank never signals at entry (the test hook): every rank's
    CTA 0 waits out a 20 ms limit, watchdog bit 3 is set and the launch
    returns; after the pads are zeroed the next call is correct."""
    import torch
    N, T, H, dt = 4, 300, 2048, "bf16"
    d = _inputs(N, T, H, dt, seed=5)
    bufs, res, g, pads = _device_group(d, N, T, H, dt, True)
    assert rarn.library().rarn_test_stall(stall_rank, 20_000_000) == 0
    rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) & 8
    for p in pads:
        p.zero_()
    bufs, res, g, _ = _device_group(d, N, T, H, dt, False)
    ref = oracle.tp_reduce_add_rms_norm([d["partials"][q] for q in range(N)], d["residual"],
                                        d["gamma"], EPS, dt)
    rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    _check(bufs, res, ref, N, T, dt, "after a reported timeout")


def test_tp_full_size_sampled():
    """Eight ranks over the reduce configuration's shape, [8192, 8192] bf16,
    with the barrier: sampled rows of every rank's buffer against the oracle's
    reduce over the same rows (the tensor-parallel form computes the reduce
    form with R = N, pinned), the residual rows of every rank."""
    import torch
    N, T, H, dt = 8, 8192, 8192, "bf16"
    rows = np.unique(np.concatenate([np.linspace(0, T - 1, 40).astype(int),
                                     [rarn.tp_rows(T, N, q)[0] for q in range(N)]]))
    w = W.workload("reduce_add_rms_norm", dt, T, H, R=N, eps=EPS, seed=3,
                   partial_std=1.0 / np.sqrt(N))
    d = W.generate(w)
    bufs, res, g, pads = _device_group(d, N, T, H, dt, True)
    rarn.tp_reduce_add_rms_norm_world(bufs, res, g, EPS, T, signals=pads)
    torch.cuda.synchronize()
    assert rarn.watchdog(clear=True) == 0
    ref = oracle.reduce_add_rms_norm(np.ascontiguousarray(d["partials"][:, rows]),
                                     np.ascontiguousarray(d["residual"][rows]), d["gamma"], EPS,
                                     dt)
    for q in range(N):
        assert_y_close(to_host(bufs[q][rows], dt), ref.y, dt, f"rank {q}'s buffer")
    for i, t in enumerate(rows):
        q = next(q for q in range(N) if rarn.tp_rows(T, N, q)[0] <= t < rarn.tp_rows(T, N, q)[1])
        r0 = rarn.tp_rows(T, N, q)[0]
        assert_bits_equal(to_host(res[q][t - r0], dt), ref.residual[i], f"row {t} residual")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ipc_rank(rank, world, port, q):
    """One rank of the two-process test (a spawned process)."""
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import torch
        import torch.distributed as dist

        import oracle as orc
        from gpu_util import assert_bits_equal as abe
        from gpu_util import assert_y_close as ayc
        from gpu_util import to_device as td
        from gpu_util import to_host as th
        import residual_add_rmsnorm_gb300 as rarn_mod
        from residual_add_rmsnorm_gb300.tp import TPGroup
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        N, T, H, dt = world, 96, 4096, "bf16"
        d = _inputs(N, T, H, dt, seed=11)
        ref = orc.tp_reduce_add_rms_norm([d["partials"][k] for k in range(N)], d["residual"],
                                         d["gamma"], EPS, dt)
        # with signal pads the two ranks' calls would wait on each other on one
        # GPU: the per-rank entry point refuses that before launching anything
        probe = TPGroup(T, H, dt, "cuda:0", signals=True)
        r0_, r1_ = probe.rows
        try:
            probe(torch.zeros(r1_ - r0_, H, dtype=torch.bfloat16, device="cuda"),
                  torch.ones(H, dtype=torch.bfloat16, device="cuda"), EPS)
            raise AssertionError("a barrier between ranks on one GPU was not refused")
        except rarn_mod.RarnError as e:
            assert e.status == 2, e
        dist.barrier()
        probe.close()
        grp = TPGroup(T, H, dt, "cuda:0", signals=False)
        grp.buffer.copy_(td(d["partials"][rank], dt))
        r0, r1 = grp.rows
        res = td(np.ascontiguousarray(d["residual"][r0:r1]), dt)
        g = td(d["gamma"], dt)
        torch.cuda.synchronize()
        dist.barrier()          # every rank's partial is in its buffer
        grp(res, g, EPS)
        torch.cuda.synchronize()
        dist.barrier()          # every rank has written its rows of y everywhere
        ayc(th(grp.buffer, dt), ref.ys[rank], dt, f"rank {rank}'s buffer")
        abe(th(res, dt), ref.residual[r0:r1], f"rank {rank} residual")
        dist.barrier()          # the peers are done with this rank's buffer
        grp.close()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent
        q.put((rank, f"{type(e).__name__}: {e}"))


def test_tp_two_processes_share_buffers_by_ipc():
    """Two processes on this GPU, each with its own buffer: the handles go
    through a gloo process group, each process opens the other's buffer, and
    each rank's call (ordered by host barriers, no signal pads) leaves y for
    all rows in both buffers."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ipc_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
    assert out == [(0, "ok"), (1, "ok")], out
    assert [p.exitcode for p in procs] == [0, 0]
