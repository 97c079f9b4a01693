"""The N > 1 host logic of bench.py on CPU: two gloo ranks, rank environment,
barrier and max-over-ranks timing, and the reference arm printing only on
rank 0.  No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    r, lr, w = bench.dist_env()
    bench.dist_init(w, use_cuda=False)
    bench.barrier()
    m = bench.max_over_ranks(float(10 + rank))
    q.put((r, lr, w, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 0, 2, 11.0), (1, 1, 2, 11.0)]


def test_reference_arm_two_ranks_prints_once():
    """torchrun-style launch of the reference arm: rank 0 prints one JSON line
    with the oracle's throughput; rank 1 exits 0 without work."""
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   LOCAL_RANK=str(r), WORLD_SIZE="2")
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "2", "--warmup", "1", "--workload", "plain_f32_T512_H2048"],
            env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    assert [p.returncode for p in procs] == [0, 0], outs
    lines0 = [ln for ln in outs[0][0].splitlines() if ln.startswith("{")]
    lines1 = [ln for ln in outs[1][0].splitlines() if ln.startswith("{")]
    assert len(lines0) == 1 and not lines1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
