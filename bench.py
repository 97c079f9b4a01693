#!/usr/bin/env python
"""Throughput of the GB300 RMSNorm library: achieved HBM GB/s and rows/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of the whole path -- reduce the R = 8 partial buffers,
add the residual, write it back, normalise, weight, write y -- over one batch
of the headline workload (reduce + residual + RMSNorm, bf16 storage,
partials [8, 8192, 8192], residual [8192, 8192]).  Its 1.3 GB of inputs are
ten times the L2, so consecutive steps read cold data without a flush.  The
other configurations of the method are timed as well and reported under
"per_config": CUDA-graph replays of launches that cycle through enough input
copies to cover twice the L2 (no host overhead, cold L2).

Rank 0 prints one JSON line.  Under torchrun each rank runs its own replica on
its own GPU (rows are independent, there is no exchange step): weak scaling,
value = all ranks' bytes / the slowest rank's time.

``--impl reference`` times the CPU oracle (the method's plain definition, in
C, binary64) on the host cores over bounded row samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "reduce8_bf16_T8192_H8192"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _configs():
    from residual_add_rmsnorm_gb300 import workloads as W
    return W.CONFIGS + W.EXTENDED + W.GEMM_CONFIGS + W.GEMM_WIDER


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=[w.name for w in _configs()] + [FP8IN_NAME, TP_NAME],
                    help="the timed configuration; a widened workload (row strides, fp32 "
                         "residual, 8-bit output or partials) has no host-buffer (e2e) or CPU "
                         "leg")
    ap.add_argument("--path", choices=["auto", "rows", "stream", "cluster"], default="auto",
                    help="kernel family (default: the library's own choice)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of untimed back-to-back steps after the timed ones, over "
                         "which nvidia-smi samples the clocks")
    ap.add_argument("--config-clock-window", type=float, default=0.5,
                    help="seconds of untimed replays per configuration for its clock record")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier and max only)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def dist_init(world, use_cuda):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend="nccl" if use_cuda else "gloo")


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(v: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def nvsmi_id(props, fallback: int) -> str:
    """The `nvidia-smi -i` identifier of a torch device: its UUID as
    nvidia-smi prints it ("GPU-..."), else the CUDA index."""
    gpu_id = str(getattr(props, "uuid", fallback))
    if gpu_id and not gpu_id.startswith("GPU-") and "-" in gpu_id:
        gpu_id = "GPU-" + gpu_id
    return gpu_id


def parse_clock_line(line: str):
    """One nvidia-smi sample: (epoch seconds, SM MHz, max SM MHz, active
    throttle reasons) or None.  nvidia-smi prints local time."""
    import datetime
    cols = [c.strip() for c in line.split(",")]
    if len(cols) != len(CLOCK_FIELDS):
        return None
    try:
        ts = datetime.datetime.strptime(cols[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        sm, smax = float(cols[1]), float(cols[2])
    except ValueError:
        return None
    reasons = {n for n, v in zip(REASONS, cols[5:]) if v.lower() == "active"}
    return ts, sm, smax, reasons


def clock_stats(samples) -> dict:
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(s[1] for s in samples),
            "sm_max_mhz": max(s[2] for s in samples),
            "reasons": sorted(set().union(*(s[3] for s in samples))), "samples": len(samples)}


class ClockSampler:
    """nvidia-smi sampling every 100 ms for the whole measurement; named
    phases (wall-clock intervals) select the samples taken while a given
    kernel ran."""

    def __init__(self, gpu_id: str, interval_ms: int = 100):
        self.proc = None
        self.path = None
        self.phases = {}
        try:
            fd, self.path = tempfile.mkstemp(prefix="rarn_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_ready(self, timeout_s: float = 5.0) -> None:
        """Block until nvidia-smi has written its first sample (it starts in a
        few hundred ms), so that the first phase is not missed."""
        t_end = time.time() + timeout_s
        while self.proc is not None and time.time() < t_end:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def begin(self, name: str) -> None:
        self.phases[name] = [time.time(), None]

    def end(self, name: str) -> None:
        if name in self.phases:
            self.phases[name][1] = time.time()

    def stop(self) -> dict:
        """Stop sampling; every phase's statistics (None without nvidia-smi)."""
        if self.proc is None:
            return {}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            samples = [s for s in map(parse_clock_line, f) if s]
        os.unlink(self.path)
        out = {}
        for name, (t0, t1) in self.phases.items():
            t1 = t1 if t1 is not None else time.time()
            out[name] = clock_stats([s for s in samples if t0 <= s[0] <= t1])
        return out


def hold_clock_window(fn, seconds: float, sync_every: int = 50) -> int:
    """Keep launching fn() back to back for about `seconds` of wall time (an
    untimed window in which nvidia-smi samples the clocks this load runs
    at); returns the launches made."""
    import torch
    n = 0
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(sync_every):
            fn()
        n += sync_every
        torch.cuda.synchronize()
    return n


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def to_device(bits, dtype, device):
    import numpy as np
    import torch
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(bits, np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
        t = t.view({"f16": torch.float16, "bf16": torch.bfloat16}[dtype])
    return t.to(device)


def kernel_source_sha(files=None) -> str:
    """sha256 over the named kernel source files (default: all of csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "residual_add_rmsnorm_gb300", "csrc")
    names = sorted(files) if files else sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def configs_summary(per_config: dict, peak: float) -> dict:
    """The method's configurations in a compact form: per workload
    [us per launch, GB/s, fraction of the measured peak, fraction of the
    nominal 8 TB/s, launch floor us (latency-bound ones), median SM MHz]."""
    from residual_add_rmsnorm_gb300 import workloads as W
    out = {"fields": ["us", "GB/s", "frac_measured", "frac_8TBps", "floor_us", "sm_mhz"]}
    for w in W.CONFIGS:
        e = per_config.get(w.name)
        if not e:
            continue
        f = e.get("floor_us")
        out[w.name] = [round(e["us_per_launch"], 2), round(e["gbs"], 0),
                       round(e["gbs"] / peak, 3), round(e["gbs"] / NOMINAL_HBM_GBS, 3),
                       None if f is None else round(f, 2), e.get("sm_mhz")]
    return out


def measured_hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            v = json.load(f).get("hbm_gbs")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload: str, plan_text: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel (the files listed in the entry) for
    this workload and plan; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    for e in data.get("entries", []):
        if (e.get("workload") == workload and e.get("plan") == plan_text
                and e.get("source_sha") == kernel_source_sha(e.get("source_files"))):
            return e.get("dram_bytes_per_launch")
    return None


E2E_HOW = ("host-buffer entry point: the kernel reads the inputs from and writes the outputs "
           "to pinned host memory (no staging copies)")


def plan_of(w, rarn) -> str:
    """The library's plan text for workload w (auto path unless forced)."""
    R = w.R if w.op == "reduce_add_rms_norm" else 1
    if w.qfmt:
        return rarn.plan_fp8(w.op, w.T, w.H, R, w.dtype)
    return rarn.plan(w.op, w.T, w.H, R, w.dtype, rdtype=w.res_dtype)


def make_call(w, tensors, rarn):
    """The public call for workload w on device tensors: the dense entry
    points, or the general ones for row-strided layouts / a binary32
    residual."""
    eps = w.eps
    general = w.row_stride != w.H or w.res_dtype != w.dtype
    if w.qfmt:  # 8-bit output: codes in y, scale in "scale"
        y, sc, g, f, m = tensors["y"], tensors["scale"], tensors["gamma"], w.qfmt, w.qmode
        if w.op == "rms_norm":
            x = tensors["x"]
            return lambda: rarn.rms_norm_fp8(x, g, eps, y, sc, f, m)
        r = tensors["residual"]
        if w.op == "fused_add_rms_norm":
            x = tensors["x"]
            return lambda: rarn.fused_add_rms_norm_fp8(x, r, g, eps, y, sc, f, m)
        p = tensors["partials"]
        return lambda: rarn.reduce_add_rms_norm_fp8(p, r, g, eps, y, sc, f, m)
    if w.op == "rms_norm":
        x, g, y = tensors["x"], tensors["gamma"], tensors["y"]
        if general:
            return lambda: rarn.rms_norm_ex(x, g, eps, out=y)
        return lambda: rarn.rms_norm(x, g, eps, out=y)
    if w.op == "fused_add_rms_norm":
        x, r, g, y = tensors["x"], tensors["residual"], tensors["gamma"], tensors["y"]
        if general:
            return lambda: rarn.fused_add_rms_norm_ex(x, r, g, eps, out=y)
        return lambda: rarn.fused_add_rms_norm(x, r, g, eps, out=y)
    p, r, g, y = tensors["partials"], tensors["residual"], tensors["gamma"], tensors["y"]
    if general:
        return lambda: rarn.reduce_add_rms_norm_ex(p, r, g, eps, out=y)
    return lambda: rarn.reduce_add_rms_norm(p, r, g, eps, out=y)


def device_tensors(w, data, device):
    """Inputs and an output buffer on the device; with a row stride, each
    [T, H] operand is a view into a [T, row_stride] allocation."""
    import torch
    ld = w.row_stride
    t = {}
    for k, v in data.items():
        dt = w.res_dtype if k == "residual" else w.dtype
        dense = to_device(v, dt, device)
        if ld != w.H and k != "gamma":
            shape = dense.shape[:-1] + (ld,)
            full = torch.empty(shape, dtype=dense.dtype, device=device)
            view = full[..., :w.H]
            view.copy_(dense)
            t[k] = view
        else:
            t[k] = dense
    ref = t.get("x", t.get("residual"))
    if w.qfmt:
        t["y"] = torch.empty((w.T, ld), dtype=torch.uint8, device=device)[:, :w.H]
        t["scale"] = (torch.full((1,), w.qscale, dtype=torch.float32, device=device)
                      if w.qmode == "tensor" else
                      torch.empty(w.T, dtype=torch.float32, device=device))
    elif ld != w.H:
        t["y"] = torch.empty((w.T, ld), dtype=to_device(data["gamma"], w.dtype, device).dtype,
                             device=device)[:, :w.H]
    else:
        t["y"] = torch.empty(ref.shape, dtype=to_device(data["gamma"], w.dtype, device).dtype,
                             device=device)
    return t


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_call(w, d, threads=0):
    import oracle
    if w.op == "rms_norm":
        return oracle.rms_norm(d["x"], d["gamma"], w.eps, w.dtype, threads=threads)
    if w.op == "fused_add_rms_norm":
        return oracle.fused_add_rms_norm(d["x"], d["residual"], d["gamma"], w.eps, w.dtype,
                                         threads=threads)
    return oracle.reduce_add_rms_norm(d["partials"], d["residual"], d["gamma"], w.eps, w.dtype,
                                      threads=threads)


def row_bytes(w) -> int:
    from residual_add_rmsnorm_gb300 import workloads as W
    return W.ELEM_SIZE[w.dtype] * w.H * (w.n_inputs + w.n_outputs)


def cpu_baseline(w, target_s: float) -> dict:
    """The oracle as it stands on the host cores, on the first rows of the
    workload, repeated until about target_s seconds of wall time."""
    from residual_add_rmsnorm_gb300 import workloads as W
    rows = min(w.T, 256)
    d = W.generate(w, rows=(0, rows))
    t0 = time.perf_counter()
    r = oracle_call(w, d)
    one = time.perf_counter() - t0
    reps = max(1, min(200, int(target_s / max(one, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(reps):
        r = oracle_call(w, d)
    el = time.perf_counter() - t0
    nbytes = rows * row_bytes(w) * reps
    out = {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": r.threads, "kind": "oracle",
           "sample": f"rows 0..{rows - 1} of {w.name}, {reps} repetitions, {el:.1f} s",
           "rows_per_s": rows * reps / el}
    # the same oracle on one core, on fewer rows
    rows1 = min(w.T, 32)
    d1 = W.generate(w, rows=(0, rows1))
    t0 = time.perf_counter()
    oracle_call(w, d1, threads=1)
    one = time.perf_counter() - t0
    reps1 = max(1, min(200, int(target_s / 3 / max(one, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(reps1):
        oracle_call(w, d1, threads=1)
    el1 = time.perf_counter() - t0
    out["value_1core"] = rows1 * row_bytes(w) * reps1 / el1 / 1e9
    out["rows_per_s_1core"] = rows1 * reps1 / el1
    out["sample_1core"] = f"rows 0..{rows1 - 1} of {w.name}, {reps1} repetitions, {el1:.1f} s"
    return out


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    from residual_add_rmsnorm_gb300 import workloads as W
    w = W.BY_NAME.get(args.workload)
    if w is None or w not in W.CONFIGS:
        raise SystemExit("the reference arm times the method's configurations only")
    rows = min(w.T, 128)
    samples = []
    nblocks = max(1, w.T // rows)
    cache = {}

    def sample(i):
        b = (i % min(nblocks, 4)) * rows
        if b not in cache:
            cache[b] = W.generate(w, rows=(b, b + rows))
        return cache[b]

    threads = 0
    for i in range(args.warmup):
        oracle_call(w, sample(i))
    for i in range(args.steps):
        d = sample(i)
        t0 = time.perf_counter()
        r = oracle_call(w, d)
        samples.append(time.perf_counter() - t0)
        threads = r.threads
    el = sum(samples)
    nbytes = rows * row_bytes(w) * args.steps
    value = nbytes / el / 1e9
    line = {
        "impl": "reference", "metric": "achieved HBM GB/s (algorithmic bytes / time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "op": w.op, "storage": w.dtype, "T": w.T, "H": w.H,
                   "R": w.R, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of {w.name} per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU measurement
# ---------------------------------------------------------------------------

def time_steps(call, steps, warmup, stream, sampler=None, window_s=0.0):
    """ms for exactly `steps` calls between CUDA events on `stream`, after
    `warmup` untimed calls, with a barrier and a synchronize on both sides.
    With a sampler, the phase "timed" covers the timed calls and the phase
    "load" also an untimed window of `window_s` seconds of the same calls
    right after them (a timed region of a few ms is shorter than the
    sampling interval)."""
    import torch
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.begin("load")
        sampler.begin("timed")
    start.record(stream)
    for _ in range(steps):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.end("timed")
        if window_s > 0:
            hold_clock_window(call, window_s)
        sampler.end("load")
    barrier()
    torch.cuda.synchronize()
    return start.elapsed_time(end)  # ms


def line_clocks(phases: dict, window_s: float) -> dict | None:
    """The JSON line's clock record: samples over the timed steps and the
    untimed window of the same steps right after them."""
    if not phases:
        return None
    load = dict(phases.get("load") or clock_stats([]))
    load["samples_in_timed_region"] = (phases.get("timed") or {}).get("samples", 0)
    load["window_s"] = window_s
    load["how"] = ("nvidia-smi every 100 ms over the timed steps and a window of the same "
                   "back-to-back steps right after them")
    return load


def time_graph(w, data, device, l2_bytes, min_launches=200, sampler=None, hold_s=0.0):
    """Per-launch device time of one configuration without host overhead and
    with a cold L2: enough copies of the inputs and outputs to cover 2 x L2
    are launched round-robin inside one CUDA graph, so no launch finds its
    data in L2 (unless one copy alone is smaller than L2 and the graph wraps
    around within it -- the copies are cycled in order, so each is evicted
    before its next use).  Returns (us per launch, copies, launches)."""
    import math

    import torch

    import residual_add_rmsnorm_gb300 as rarn
    footprint = w.algorithmic_bytes()
    copies = max(1, min(64, math.ceil(2 * l2_bytes / footprint)))
    sets = [device_tensors(w, data, device) for _ in range(copies)]
    calls = [make_call(w, t, rarn) for t in sets]
    per_pass = copies
    passes = max(1, math.ceil(min_launches / per_pass))
    # keep huge configurations short: at most ~40 GB of traffic per replay
    passes = max(1, min(passes, int(40e9 // (footprint * copies))))
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for c in calls:
            c()
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(passes):
            for c in calls:
                c()
    n = passes * per_pass
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(device)
    times = []
    for _ in range(3):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    if sampler and hold_s > 0:  # clocks under this load, untimed
        sampler.begin(w.name)
        hold_clock_window(graph.replay, hold_s, sync_every=max(1, int(2000 // n)))
        sampler.end(w.name)
    del graph, sets, calls
    return 1e3 * statistics.median(times) / n, copies, n


def plan_field(plan: str, key: str) -> int | None:
    import re
    m = re.search(rf"\b{key}=(\d+)", plan)
    return int(m.group(1)) if m else None


def time_floor(w, plan: str, device, l2_bytes, min_launches=200):
    """The launch floor of a configuration: its plan's grid and block of the
    library's empty kernel (one row per CTA prefetched into L2, the
    dependency wait and the trigger, the same PDL setting), timed like the
    configuration itself (CUDA graph, rows cycled so each launch prefetches
    cold rows).  None if the plan has no grid."""
    import math

    import torch

    import residual_add_rmsnorm_gb300 as rarn
    from residual_add_rmsnorm_gb300 import workloads as W
    grid, block = plan_field(plan, "grid"), plan_field(plan, "block")
    if not grid or not block:
        return None
    # a CTA's first row: its inputs (x, the residual, the partials)
    row_bytes = (w.n_inputs * W.ELEM_SIZE[w.dtype] * w.H + 15) // 16 * 16
    row_bytes = min(row_bytes, 1 << 20)
    copies = max(1, min(64, math.ceil(2 * l2_bytes / (grid * row_bytes))))
    buf = torch.empty(copies * grid * row_bytes, dtype=torch.uint8, device=device)
    views = [buf[i * grid * row_bytes:(i + 1) * grid * row_bytes] for i in range(copies)]
    passes = max(1, math.ceil(min_launches / copies))
    for v in views:
        rarn.launch_floor(grid, block, v, row_bytes)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(passes):
            for v in views:
                rarn.launch_floor(grid, block, v, row_bytes)
    n = passes * copies
    graph.replay()
    torch.cuda.synchronize(device)
    times = []
    for _ in range(3):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    del graph, views, buf
    return 1e3 * statistics.median(times) / n


def measured_tensor_peak():
    """Dense bf16 TFLOP/s measured on this machine's GPUs (burst: a kernel timed
    alone), else the fallback."""
    try:
        with open(PEAKS_FILE) as f:
            v = json.load(f).get("bf16_tflops")
        if v:
            return float(v), "measured bf16_tflops (burst)"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def _graph_us(fn, launches=10, reps=3, sampler=None, phase=None, hold_s=0.0):
    """Per-launch device time of fn() replayed in a CUDA graph (best of reps);
    with a sampler, the graph is then replayed untimed for hold_s seconds
    under the phase name, so the clocks of this load are sampled."""
    import torch
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(launches):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        e.synchronize()
        t = 1e3 * s.elapsed_time(e) / launches
        best = t if best is None else min(best, t)
    if sampler and phase and hold_s > 0:
        sampler.begin(phase)
        hold_clock_window(graph.replay, hold_s, sync_every=5)
        sampler.end(phase)
    return best


def time_gemm(gw, device, rarn, sampler=None, hold_s=0.0):
    """The GEMM-producer form: one tcgen05 kernel (matrix product, residual
    add, RMSNorm) timed against the unfused sequence the same library offers
    a user (cuBLAS product through torch.matmul, then the fused norm kernel);
    TFLOP/s of the 2 T H K product against the measured tensor peak."""
    import torch
    from residual_add_rmsnorm_gb300 import workloads as W
    d = W.generate_gemm(gw)
    a, w, r, g = (to_device(d[k], gw.dtype, device) for k in ("a", "w", "residual", "gamma"))
    y = torch.empty_like(r)
    part = torch.empty_like(r)
    us = _graph_us(lambda: rarn.gemm_add_rms_norm(a, w, r, g, gw.eps, out=y), sampler=sampler,
                   phase=gw.name, hold_s=hold_s)
    us_mm = _graph_us(lambda: torch.matmul(a, w.t(), out=part))
    us_unfused = _graph_us(lambda: (torch.matmul(a, w.t(), out=part),
                                    rarn.fused_add_rms_norm(part, r, g, gw.eps, out=y)))
    peak, kind = measured_tensor_peak()
    tflops = gw.flops() / (us / 1e6) / 1e12
    return {"kind": "widened (GEMM producer)", "us_per_launch": us, "tflops": tflops,
            "frac_of_tensor_peak": tflops / peak, "tensor_peak": peak, "peak_source": kind,
            "gbs_algorithmic": gw.algorithmic_bytes() / (us / 1e6) / 1e9,
            "unfused_us": us_unfused, "cublas_matmul_us": us_mm,
            "timing": "CUDA graph of 10 launches, best of 3 (operands L2-resident after the "
                      "first launch)",
            "plan": rarn.plan_gemm(gw.T, gw.H, gw.K, gw.dtype, num_sms=0)}


FP8IN_NAME = "reduce8_e4m3in_bf16_T8192_H8192"
TP_NAME = "tp8_world_bf16_T8192_H8192"


def tp_tensors(device, N=8, T=8192, H=8192):
    """The tensor-parallel form over N ranks' buffers held on this one GPU
    (the reduce configuration's shape): N partials N(0, 1/N) bf16, the
    residual N(0, 1) split into the ranks' row blocks, gamma U(0.5, 1.5),
    zeroed signal pads; and the algorithmic bytes of one call (every rank's
    row block read from every buffer, the residual read and written, y
    written into every buffer, gamma)."""
    import torch

    import residual_add_rmsnorm_gb300 as rarn
    gen = torch.Generator(device=device).manual_seed(0)
    bufs = [(torch.randn(T, H, device=device, generator=gen) / N ** 0.5).to(torch.bfloat16)
            for _ in range(N)]
    res = []
    for q in range(N):
        r0, r1 = rarn.tp_rows(T, N, q)
        res.append(torch.randn(r1 - r0, H, device=device, generator=gen).to(torch.bfloat16))
    g = (torch.rand(H, device=device, generator=gen) + 0.5).to(torch.bfloat16)
    pads = [torch.zeros(rarn.TP_SIGNAL_BYTES // 4, dtype=torch.int32, device=device)
            for _ in range(N)]
    alg = (N * T * H + 2 * T * H + N * T * H) * 2 + H * 2
    return bufs, res, g, pads, alg


def time_tp(device, rarn, N=8, T=8192, H=8192, sampler=None, hold_s=0.0):
    """Every rank's part in one launch with the signal-pad barrier: the
    data path and the synchronisation on this GPU's memory (no NVLink
    traffic: an emulation of N GPUs, not a multi-GPU measurement)."""
    import torch
    bufs, res, g, pads, alg = tp_tensors(device, N, T, H)
    us = _graph_us(lambda: rarn.tp_reduce_add_rms_norm_world(bufs, res, g, 1e-6, T,
                                                             signals=pads),
                   sampler=sampler, phase=TP_NAME, hold_s=hold_s)
    peak, _ = measured_hbm_peak()
    gbs = alg / (us / 1e6) / 1e9
    del bufs, res, pads
    torch.cuda.empty_cache()
    return {"kind": "widened (tensor-parallel, N ranks' buffers on one GPU)",
            "us_per_launch": us, "gbs": gbs, "rows_per_s": T / (us / 1e6),
            "frac_of_peak": gbs / peak, "algorithmic_bytes": alg, "ranks": N,
            "timing": "CUDA graph of 10 launches, best of 3 (inputs larger than L2)",
            "plan": rarn.plan_tp(T, H, N, "bf16", True, 0, 0) + " barrier=signal pads"}


def fp8in_tensors(device, R=8, T=8192, H=8192):
    """Seeded synthetic inputs of the reduce over 8-bit partials: codes
    N(0, 1) scaled to the e4m3 range and cast to e4m3, scales U(0.5, 1.5),
    residual N(0, 1) bf16, gamma U(0.5, 1.5) bf16; and the algorithmic bytes
    of one call (R T H codes, residual read and written, y, gamma, scales)."""
    import torch
    gen = torch.Generator(device=device).manual_seed(0)
    codes = torch.empty(R, T, H, dtype=torch.uint8, device=device)
    for r in range(R):
        v = torch.randn(T, H, device=device, generator=gen) * (448.0 / 16)
        codes[r] = v.to(torch.float8_e4m3fn).view(torch.uint8)
        del v
    scales = torch.rand(R, device=device, generator=gen) + 0.5
    res = torch.randn(T, H, device=device, generator=gen).to(torch.bfloat16)
    g = (torch.rand(H, device=device, generator=gen) + 0.5).to(torch.bfloat16)
    return codes, scales, res, g, R * T * H + 3 * T * H * 2 + H * 2 + R * 4


def fp8in_plan(device, rarn, R=8, T=8192, H=8192) -> str:
    """The library's description of the kernel the 8-bit-partials call takes
    on this device (its SM count and opt-in shared memory per CTA)."""
    import torch
    props = torch.cuda.get_device_properties(device)
    smem = getattr(props, "shared_memory_per_block_optin", 0) or 232448
    return rarn.plan_fp8in(T, H, R, "bf16", True, props.multi_processor_count, smem)


def time_fp8in(device, rarn, R=8, T=8192, H=8192, sampler=None, hold_s=0.0):
    """The reduce over 8-bit partials on the headline shape; the inputs
    (0.9 GB) exceed L2, so launches read cold data."""
    import torch
    codes, scales, res, g, alg = fp8in_tensors(device, R, T, H)
    y = torch.empty_like(res)
    us = _graph_us(lambda: rarn.reduce_add_rms_norm_fp8in(codes, scales, res, g, 1e-6, "e4m3",
                                                          out=y),
                   sampler=sampler, phase=FP8IN_NAME, hold_s=hold_s)
    peak, _ = measured_hbm_peak()
    gbs = alg / (us / 1e6) / 1e9
    del codes, res, y
    torch.cuda.empty_cache()
    return {"kind": "widened (8-bit partials)", "us_per_launch": us, "gbs": gbs,
            "rows_per_s": T / (us / 1e6), "frac_of_peak": gbs / peak, "algorithmic_bytes": alg,
            "timing": "CUDA graph of 10 launches, best of 3 (inputs larger than L2)",
            "plan": fp8in_plan(device, rarn, R, T, H)}


def main_fp8in(args, device, rank, world):
    """The reduce over 8-bit partials as the timed step (one launch per
    step; inputs resident in HBM and larger than L2).  No host-buffer entry
    point and no oracle leg for this form."""
    import torch

    import residual_add_rmsnorm_gb300 as rarn
    codes, scales, res, g, alg = fp8in_tensors(device)
    plan = fp8in_plan(device, rarn)
    y = torch.empty_like(res)
    call = lambda: rarn.reduce_add_rms_norm_fp8in(codes, scales, res, g, 1e-6, "e4m3", out=y)
    stream = torch.cuda.current_stream(device)
    sampler = ClockSampler(nvsmi_id(torch.cuda.get_device_properties(device), device.index or 0))
    sampler.wait_ready()
    ms = time_steps(call, args.steps, args.warmup, stream, sampler, args.clock_window)
    clocks = line_clocks(sampler.stop(), args.clock_window)
    ms = max_over_ranks(ms, device)
    peak, kind = measured_hbm_peak()
    gbs = world * alg * args.steps / (ms / 1e3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": "achieved HBM GB/s (algorithmic bytes / time)", "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": FP8IN_NAME, "R": 8, "T": 8192, "H": 8192, "format": "e4m3",
                   "storage": "bf16", "plan": plan,
                   "l2": "inputs larger than L2 (0.9 GB)", "pdl": not args.no_pdl},
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peak, "unit": "GB/s",
                     "frac": gbs / world / peak,
                     "traffic": ncu_traffic(FP8IN_NAME, plan), "peak_source": kind},
        "cpu_baseline": None,
        "e2e": {"value": None, "unit": "GB/s",
                "note": "no host-buffer entry point for the 8-bit-partials form"},
        "clocks": clocks, "gpu_launches": args.steps, "watchdog": rarn.watchdog(clear=True),
    }
    print(json.dumps(line), flush=True)


def main_tp(args, device, rank, world):
    """The tensor-parallel form as the timed step: eight ranks' buffers on
    this GPU, every rank's part in one launch with the barrier (one launch
    per step; inputs resident in HBM, larger than L2).  No host-buffer entry
    point and no oracle leg for this form."""
    import torch

    import residual_add_rmsnorm_gb300 as rarn
    N, T, H = 8, 8192, 8192
    bufs, res, g, pads, alg = tp_tensors(device, N, T, H)
    call = lambda: rarn.tp_reduce_add_rms_norm_world(bufs, res, g, 1e-6, T, signals=pads)
    stream = torch.cuda.current_stream(device)
    sampler = ClockSampler(nvsmi_id(torch.cuda.get_device_properties(device), device.index or 0))
    sampler.wait_ready()
    ms = time_steps(call, args.steps, args.warmup, stream, sampler, args.clock_window)
    clocks = line_clocks(sampler.stop(), args.clock_window)
    ms = max_over_ranks(ms, device)
    peak, kind = measured_hbm_peak()
    gbs = world * alg * args.steps / (ms / 1e3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": "achieved HBM GB/s (algorithmic bytes / time)", "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": TP_NAME, "ranks": N, "T": T, "H": H, "storage": "bf16",
                   "plan": rarn.plan_tp(T, H, N, "bf16", True, 0, 0) + " barrier=signal pads",
                   "l2": "inputs larger than L2 (1.2 GB)", "pdl": not args.no_pdl,
                   "note": "the N ranks' buffers are on this one GPU: no NVLink traffic"},
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peak, "unit": "GB/s",
                     "frac": gbs / world / peak, "traffic": ncu_traffic(TP_NAME, "tp.world"),
                     "peak_source": kind},
        "cpu_baseline": None,
        "e2e": {"value": None, "unit": "GB/s",
                "note": "no host-buffer entry point for the tensor-parallel form"},
        "clocks": clocks, "gpu_launches": args.steps, "watchdog": rarn.watchdog(clear=True),
    }
    print(json.dumps(line), flush=True)


def e2e_steps(w, data, steps, device, stream):
    """End to end through the public host-buffer API: the inputs start in
    pinned host memory and the outputs end there.  Each step is one call of
    the *_host entry point, whose kernel reads the step's inputs from host
    memory and writes y and the residual back to it over the host link; no
    staging copy and no device buffer is involved.  Returns (ms for `steps`
    steps, host->device bytes per step, device->host bytes per step)."""
    import residual_add_rmsnorm_gb300 as rarn
    hin = {k: to_device(v, w.dtype, "cpu").pin_memory() for k, v in data.items()}
    ref = hin.get("x", hin.get("residual"))
    hy = ref.new_empty(ref.shape).pin_memory()
    if w.op == "rms_norm":
        call = lambda: rarn.rms_norm_host(hin["x"], hin["gamma"], w.eps, out=hy, device=device)
    elif w.op == "fused_add_rms_norm":
        call = lambda: rarn.fused_add_rms_norm_host(hin["x"], hin["residual"], hin["gamma"],
                                                    w.eps, out=hy, device=device)
    else:
        call = lambda: rarn.reduce_add_rms_norm_host(hin["partials"], hin["residual"],
                                                     hin["gamma"], w.eps, out=hy, device=device)
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = hy.numel() * hy.element_size() * w.n_outputs
    ms = time_steps(call, steps, 2, stream)
    return ms, h2d, d2h


def main_gemm(args, gw, device, rank, world):
    """The GEMM-producer form as the timed step: one call = the tcgen05 GEMM
    with the residual add and the norm (two kernels).  TFLOP/s of the 2 T H K
    product; inputs resident in HBM; no host-buffer or CPU leg."""
    import torch

    import residual_add_rmsnorm_gb300 as rarn
    from residual_add_rmsnorm_gb300 import workloads as W
    d = W.generate_gemm(gw)
    a, w, r, g = (to_device(d[k], gw.dtype, device) for k in ("a", "w", "residual", "gamma"))
    y = torch.empty_like(r)
    ws = torch.empty(max(rarn.gemm_workspace_bytes(gw.T, gw.H), 4) // 4, dtype=torch.float32,
                     device=device)
    call = lambda: rarn.gemm_add_rms_norm(a, w, r, g, gw.eps, out=y, workspace=ws)
    stream = torch.cuda.current_stream(device)
    sampler = ClockSampler(nvsmi_id(torch.cuda.get_device_properties(device), device.index or 0))
    sampler.wait_ready()
    ms = time_steps(call, args.steps, args.warmup, stream, sampler, args.clock_window)
    clocks = line_clocks(sampler.stop(), args.clock_window)
    ms = max_over_ranks(ms, device)
    peak, kind = measured_tensor_peak()
    tflops = world * gw.flops() * args.steps / (ms / 1e3) / 1e12
    if rank != 0:
        return
    line = {
        "metric": "achieved TFLOP/s of the product (2 T H K / time)", "value": tflops,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": gw.dtype, "data": "synthetic",
        "config": {"workload": gw.name, "T": gw.T, "H": gw.H, "K": gw.K,
                   "plan": rarn.plan_gemm(gw.T, gw.H, gw.K, gw.dtype, num_sms=0),
                   "l2": "operands L2-resident after the first step (64 MB)",
                   "pdl": not args.no_pdl},
        "roofline": {"bound": "tensor", "achieved": tflops / world, "peak": peak,
                     "unit": "TFLOP/s", "frac": tflops / world / peak, "traffic": None,
                     "peak_source": kind},
        "cpu_baseline": None,
        "e2e": {"value": None, "unit": "TFLOP/s",
                "note": "no host-buffer entry point for the GEMM form"},
        "clocks": clocks, "gpu_launches": 2 * args.steps, "watchdog": rarn.watchdog(clear=True),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        dist_init(world, use_cuda=False)
        run_reference(args)
        return
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist_init(world, use_cuda=True)

    import residual_add_rmsnorm_gb300 as rarn
    from residual_add_rmsnorm_gb300 import build as rbuild
    from residual_add_rmsnorm_gb300 import workloads as W
    rbuild.build()

    rarn.set_path(args.path)
    rarn.set_pdl(not args.no_pdl)
    gemm = {gw.name: gw for gw in W.GEMM_CONFIGS + W.GEMM_WIDER}
    if args.workload in gemm:
        main_gemm(args, gemm[args.workload], device, rank, world)
        return
    if args.workload == FP8IN_NAME:
        main_fp8in(args, device, rank, world)
        return
    if args.workload == TP_NAME:
        main_tp(args, device, rank, world)
        return
    w = W.BY_NAME[args.workload]
    data = W.generate(w)
    tensors = device_tensors(w, data, device)
    call = make_call(w, tensors, rarn)
    stream = torch.cuda.current_stream(device)
    plan_text = plan_of(w, rarn)
    dense = w in W.CONFIGS  # the forms the host-buffer entry points and the oracle leg cover

    props = torch.cuda.get_device_properties(device)
    sampler = ClockSampler(nvsmi_id(props, local_rank))
    sampler.wait_ready()
    ms = time_steps(call, args.steps, args.warmup, stream, sampler, args.clock_window)
    ms = max_over_ranks(ms, device)
    alg = w.algorithmic_bytes()
    per_launch_s = ms / 1e3 / args.steps
    value = world * alg * args.steps / (ms / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    achieved = alg / per_launch_s / 1e9

    e2e = {"value": None, "unit": "GB/s",
           "note": "no host-buffer entry point for this form (dense forms only)"}
    if dense:
        e2e_ms, h2d, d2h = e2e_steps(w, data, args.e2e_steps, device, stream)
        e2e_ms = max_over_ranks(e2e_ms, device)
        e2e = {"value": world * alg * args.e2e_steps / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "how": E2E_HOW}
    watchdog = rarn.watchdog(clear=True)

    per_config = {}
    hold = args.config_clock_window
    if not args.no_configs:
        l2 = int(getattr(props, "L2_cache_size", 128 << 20))
        del tensors, call
        torch.cuda.empty_cache()
        rarn.set_path("auto")
        for cw in W.CONFIGS + W.EXTENDED:
            cd = W.generate(cw)
            us, copies, n = time_graph(cw, cd, device, l2, sampler=sampler, hold_s=hold)
            cb = cw.algorithmic_bytes()
            gbs = cb / (us / 1e6) / 1e9
            plan = plan_of(cw, rarn)
            per_config[cw.name] = {
                "kind": "widened" if cw in W.EXTENDED else "config",
                "us_per_launch": us, "gbs": gbs, "rows_per_s": cw.T / (us / 1e6),
                "frac_of_peak": gbs / peak, "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                "algorithmic_bytes": cb,
                "timing": f"CUDA graph of {n} launches over {copies} input copies (cold L2)",
                "plan": plan}
            if cw in W.CONFIGS and cw.algorithmic_bytes() < 64e6:
                # latency-bound: the launch floor of the same grid and block
                floor = time_floor(cw, plan, device, l2)
                per_config[cw.name]["floor_us"] = floor
                per_config[cw.name]["us_above_floor"] = None if floor is None else us - floor
            del cd
            torch.cuda.empty_cache()
        # the memory-bound entries before the tensor-bound GEMM ones: right
        # after seconds of GEMMs at the power cap, the 8-bit-partials kernel
        # measured 162 us against 142 us when timed first
        per_config[FP8IN_NAME] = time_fp8in(device, rarn, sampler=sampler, hold_s=hold)
        per_config[TP_NAME] = time_tp(device, rarn, sampler=sampler, hold_s=hold)
        for gw in W.GEMM_CONFIGS + W.GEMM_WIDER:
            per_config[gw.name] = time_gemm(gw, device, rarn, sampler=sampler, hold_s=hold)
        if rarn.watchdog(clear=True):
            watchdog = 1
    phases = sampler.stop()
    clocks = line_clocks(phases, args.clock_window)
    for name, entry in per_config.items():
        st = phases.get(name)
        if st:
            entry["sm_mhz"] = st["sm_mhz"]
            entry["clock_samples"] = st["samples"]
            entry["clock_reasons"] = st["reasons"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and dense:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank != 0:
        return
    line = {
        "metric": "achieved HBM GB/s (algorithmic bytes / time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "op": w.op, "storage": w.dtype, "T": w.T, "H": w.H,
                   "R": w.R, "eps": w.eps, "rows_per_s": world * w.T * args.steps / (ms / 1e3),
                   "l2": "inputs larger than L2 (no flush between steps)",
                   "parallelism": "replicas" if world > 1 else "single",
                   "plan": plan_text, "pdl": not args.no_pdl},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(w.name, plan_text),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": alg},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": args.steps,
        "watchdog": watchdog,
        "per_config": per_config,
        # last, so that a tail of the output still carries it: every
        # configuration of the method in a few numbers
        "configs_summary": configs_summary(per_config, peak),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
