"""Host side of the tensor-parallel form, on CPU: the row partition against
the oracle's, argument checks before any CUDA call, and a two-rank gloo group
exchanging its buffers' handles (an IPC backend that stands in for CUDA IPC,
so no GPU is touched)."""
import ctypes
import os
import socket
import sys

import pytest

import oracle
import residual_add_rmsnorm_gb300 as rarn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIAS = 0, 1, 2, 3
F32, F16, BF16 = 0, 1, 2
# fake, never dereferenced device addresses: every call below fails its
# argument checks before reaching CUDA
A = 1 << 40


def test_rows_match_the_oracle():
    for N in range(1, 9):
        for T in (0, 1, 2, 7, 8, 100, 4097):
            blocks = [rarn.tp_rows(T, N, r) for r in range(N)]
            assert blocks == [oracle.tp_rows(T, N, r) for r in range(N)], (T, N)
    for bad in ((-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)):
        with pytest.raises(rarn.RarnError):
            rarn.tp_rows(*bad)


def _group(N, rank, bufs=None, sigs=None):
    g = rarn.TpGroup()
    g.world_size = N
    g.rank = rank
    for q in range(min(N, rarn.TP_MAX_RANKS)):
        g.buffers[q] = bufs[q] if bufs is not None else A + q * (1 << 32)
        if sigs is not None:
            g.signals[q] = sigs[q]
    return g


def test_tp_argument_errors():
    lib = rarn.library()
    f = lib.rarn_tp_reduce_add_rms_norm
    T, H = 64, 4096
    res, gam = A + (100 << 32), A + (101 << 32)

    def call(g, r=res, gm=gam, T=T, H=H, eps=1e-6, dt=BF16):
        return f(ctypes.byref(g) if g is not None else None, r, gm, T, H, eps, dt, None)

    assert call(None) == INVALID
    assert call(_group(0, 0)) == INVALID
    assert call(_group(9, 0)) == INVALID
    assert call(_group(4, 4)) == INVALID                      # rank out of range
    assert call(_group(2, 0), eps=-1.0) == INVALID
    assert call(_group(2, 0), dt=7) == INVALID
    assert call(_group(2, 0), r=None) == INVALID
    assert call(_group(2, 0), gm=None) == INVALID
    assert call(_group(2, 0, bufs=[A, 0])) == INVALID         # a missing buffer
    sig = [A + (200 << 32), A + (201 << 32)]
    assert call(_group(2, 0, sigs=[sig[0], 0])) == INVALID    # pads for some ranks only
    assert call(_group(2, 0), H=4092) == UNSUPPORTED           # rows not whole 16-byte packs
    assert call(_group(2, 0), H=16392) == UNSUPPORTED          # beyond 2048 packs
    assert call(_group(2, 0, bufs=[A + 8, A + (1 << 32)])) == UNSUPPORTED
    assert call(_group(2, 0, sigs=[sig[0] + 2, sig[1]])) == UNSUPPORTED
    assert call(_group(2, 0, bufs=[A, A + 1024])) == ALIAS    # two ranks' buffers overlap
    assert call(_group(2, 0), r=A + 64) == ALIAS               # residual inside a buffer
    assert call(_group(2, 0), gm=A + (1 << 32) + 16) == ALIAS
    assert call(_group(2, 0, sigs=[A + 16, sig[1]])) == ALIAS  # a pad inside a buffer
    assert call(_group(2, 0), T=0) == OK                       # nothing to do
    w = lib.rarn_tp_reduce_add_rms_norm_world
    assert w(ctypes.byref(_group(2, 0)), None, gam, T, H, 1e-6, BF16, None) == INVALID
    rp = (ctypes.c_void_p * 2)(res, 0)
    assert w(ctypes.byref(_group(2, 0)), ctypes.cast(rp, ctypes.c_void_p), gam, T, H, 1e-6,
             BF16, None) == INVALID                            # a rank's residual missing


def _plan_fields(text):
    head, *kv = text.split()
    return head, {k: int(v) for k, v in (f.split("=") for f in kv)}


# (N, H, dtype, CTAs per SM) -> whether each CTA prefetches its next row: the
# shapes of the prefetch A/B on a GB300 (two to eight ranks' buffers on one
# GPU), on the side the measurement came out
PREFETCH_CASES = [
    (1, 8192, "bf16", 1, 1), (2, 8192, "bf16", 1, 1), (3, 8192, "bf16", 1, 1),
    (4, 8192, "bf16", 1, 1), (4, 8192, "f16", 1, 1), (2, 5120, "bf16", 1, 1),
    (4, 5120, "bf16", 1, 1), (2, 4096, "f32", 1, 1), (2, 4096, "bf16", 2, 1),
    (2, 2048, "bf16", 4, 1),
    (5, 8192, "bf16", 1, 0), (6, 8192, "bf16", 1, 0), (8, 8192, "bf16", 1, 0),
    (2, 8192, "f32", 1, 0), (4, 8192, "f32", 1, 0), (4, 4096, "bf16", 2, 0),
    (8, 4096, "bf16", 2, 0), (4, 2048, "bf16", 4, 0),
]


@pytest.mark.parametrize("N,H,dt,per_sm,want", PREFETCH_CASES)
def test_plan_tp_prefetch_rule(N, H, dt, per_sm, want, tune):
    """The next-row L2 prefetch is on where an SM's loads in flight, per_sm
    CTAs x (N + 1) rows, come to at most 64 KB, or 80 KB with one CTA per
    SM; the knob forces it either way."""
    size = {"f32": 4, "f16": 2, "bf16": 2}[dt]
    inflight = per_sm * (N + 1) * H * size
    assert want == int(inflight <= 65536 or (per_sm == 1 and inflight <= 81920))
    head, f = _plan_fields(rarn.plan_tp(8192, H, N, dt, True, 152, per_sm))
    assert head == "tp.world" and f["ranks"] == N and f["blocks_per_sm"] == per_sm
    assert f["prefetch"] == want
    for v in (0, 1):
        tune(tp_prefetch=v)
        assert _plan_fields(rarn.plan_tp(8192, H, N, dt, True, 152, per_sm))[1]["prefetch"] == v


def test_plan_tp_launch_shape():
    """CTAs per rank: the SMs' resident CTAs shared among the ranks of the
    world launch (all of them for one rank's launch), at most 1024, and the
    largest row block spread evenly over as few rounds as that allows; the
    thread shape: the fewest 16-byte packs per thread (1, 2, 4) that keep a
    CTA within 512 threads."""
    for T, H, N, dt, world, sms, per_sm in [
            (8192, 8192, 8, "bf16", True, 152, 1), (8192, 4096, 8, "bf16", True, 152, 2),
            (16384, 8192, 2, "bf16", True, 152, 1), (100, 2048, 4, "f32", True, 152, 2),
            (3, 512, 8, "f16", True, 152, 4), (8192, 8192, 8, "bf16", False, 152, 1),
            (1 << 20, 1024, 1, "f32", False, 152, 8), (4097, 16384, 2, "bf16", True, 7, 1)]:
        head, f = _plan_fields(rarn.plan_tp(T, H, N, dt, world, sms, per_sm))
        assert head == ("tp.world" if world else "tp.rank")
        rows_max = -(-T // N)
        slots = max(1, min(1024, sms * per_sm // (N if world else 1)))
        rounds = -(-rows_max // slots)
        assert f["ctas"] == -(-rows_max // rounds) <= slots, (T, H, N, f)
        if world:
            assert f["ctas"] * N <= sms * per_sm or f["ctas"] == 1
        nv = H * {"f32": 4, "f16": 2, "bf16": 2}[dt] // 16
        vpt = 1 if nv <= 512 else 2 if nv <= 1024 else 4
        assert f["vpt"] == vpt, f
        assert f["block"] == (-(-nv // vpt) + 31) // 32 * 32 <= 512, f
    lib = rarn.library()
    buf = ctypes.create_string_buffer(128)
    plan = lib.rarn_plan_tp
    assert plan(64, 4096, 2, BF16, 1, 152, 1, None, 128) == INVALID
    assert plan(64, 4096, 2, BF16, 1, 152, 1, buf, 0) == INVALID
    for bad in ((0, 4096, 2, BF16), (64, 0, 2, BF16), (64, 4096, 0, BF16), (64, 4096, 9, BF16),
                (64, 4096, 2, 7)):
        assert plan(*bad, 1, 152, 1, buf, 128) == INVALID, bad
    assert plan(64, 4092, 2, BF16, 1, 152, 1, buf, 128) == UNSUPPORTED
    assert buf.value.startswith(b"none")
    assert plan(64, 16392, 2, BF16, 1, 152, 1, buf, 128) == UNSUPPORTED


def test_plan_tp_device_queries():
    """With the SM count or the occupancy left to the device, the plan query
    asks the current device: RARN_ERR_CUDA where there is none (this host),
    the same answer as the explicit form where there is one."""
    import torch
    lib = rarn.library()
    buf = ctypes.create_string_buffer(128)
    for sms, per_sm in ((0, 1), (152, 0), (0, 0)):
        st = lib.rarn_plan_tp(8192, 8192, 2, BF16, 1, sms, per_sm, buf, 128)
        if torch.cuda.is_available():
            assert st == OK and buf.value.startswith(b"tp.world"), (sms, per_sm, buf.value)
        else:
            assert st == 4, (sms, per_sm, st)   # RARN_ERR_CUDA: no device to ask
            assert lib.rarn_last_cuda_error() != 0
    # argument errors come first, device or not
    assert lib.rarn_plan_tp(8192, 8192, 9, BF16, 1, 0, 0, buf, 128) == INVALID


def test_ipc_handle_checks():
    lib = rarn.library()
    h = ctypes.create_string_buffer(rarn.IPC_HANDLE_BYTES)
    p = ctypes.c_void_p(0)
    assert lib.rarn_ipc_export(None, h) == INVALID
    assert lib.rarn_ipc_export(A, None) == INVALID
    assert lib.rarn_ipc_import(h, ctypes.byref(p)) == INVALID  # not a handle of this library
    assert lib.rarn_ipc_import(None, ctypes.byref(p)) == INVALID
    assert lib.rarn_ipc_close(A) == INVALID                     # never opened
    with pytest.raises(ValueError):
        rarn.ipc_import(b"short")


class FakeIpc:
    """Stands in for CUDA IPC: a handle carries the exporting rank and the
    address; opening one returns that address tagged with the opener."""

    def __init__(self, rank):
        self.rank = rank
        self.closed = []

    def export(self, t) -> bytes:
        return b"%d:%d" % (self.rank, t.data_ptr())

    def open(self, handle: bytes) -> int:
        src, addr = handle.split(b":")
        assert int(src) != self.rank, "a process never opens its own handle"
        return int(addr)

    def close(self, ptr: int) -> None:
        self.closed.append(ptr)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from residual_add_rmsnorm_gb300.tp import TPGroup
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ipc = FakeIpc(rank)
    g = TPGroup(11, 64, "bf16", "cpu", signals=True, ipc=ipc)
    own = (g.buffer.data_ptr(), g.pad.data_ptr())
    every = [None] * world
    dist.all_gather_object(every, own)
    rows = [None] * world
    dist.all_gather_object(rows, g.rows)
    g.close()
    q.put((rank, g.buffers, g.signals, every, rows, sorted(ipc.closed)))
    dist.destroy_process_group()


def test_two_ranks_exchange_handles_and_split_rows():
    """Each rank ends with every rank's buffer and pad in rank order (its own
    at its own index, the others opened from their handles), the ranks' row
    blocks tile 0 .. T-1 in rank order, and close() releases exactly what was
    opened."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, bufs, sigs, every, rows, closed in out:
        assert bufs == [every[0][0], every[1][0]], rank
        assert sigs == [every[0][1], every[1][1]], rank
        other = 1 - rank
        assert closed == sorted([every[other][0], every[other][1]])
        assert rows == [(0, 5), (5, 11)]
