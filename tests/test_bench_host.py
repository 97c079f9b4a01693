"""bench.py's host-side bookkeeping on CPU: the committed ncu traffic table
is well formed, names summaries that exist, and is only used for the
workload, plan and kernel sources it was captured on."""
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    import sys
    sys.path.insert(0, ROOT)
    import bench as b
    return b


def test_traffic_table_well_formed(bench):
    with open(bench.TRAFFIC_FILE) as f:
        data = json.load(f)
    names = {w.name for w in bench._configs()} | {bench.FP8IN_NAME, bench.TP_NAME}
    csrc = os.path.join(ROOT, "residual_add_rmsnorm_gb300", "csrc")
    for e in data["entries"]:
        assert e["workload"] in names, e["workload"]
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert os.path.isfile(os.path.join(ROOT, e["summary"])), e["summary"]
        for src in e["source_files"]:
            assert os.path.isfile(os.path.join(csrc, src)), src
        assert len(e["source_sha"]) == 64 and e["plan"]


def test_traffic_lookup_keys(bench, tmp_path, monkeypatch):
    """A lookup returns the bytes only for the recorded workload and plan
    while the listed sources still hash to the recorded value."""
    csrc_files = ["common.cuh"]
    entry = {"workload": "w", "plan": "p", "kernel": "k", "source_files": csrc_files,
             "source_sha": bench.kernel_source_sha(csrc_files), "dram_bytes_read": 3,
             "dram_bytes_write": 4, "dram_bytes_per_launch": 7, "summary": "s.md"}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"entries": [entry]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.ncu_traffic("w", "p") == 7
    assert bench.ncu_traffic("w", "other plan") is None
    assert bench.ncu_traffic("other", "p") is None
    entry["source_sha"] = "0" * 64
    f.write_text(json.dumps({"entries": [entry]}))
    assert bench.ncu_traffic("w", "p") is None


def test_nvsmi_id(bench):
    """nvidia-smi is given the device's UUID with its "GPU-" prefix, or the
    CUDA index when torch reports no UUID."""
    class P:
        pass
    p = P()
    assert bench.nvsmi_id(p, 3) == "3"
    p.uuid = "1a2b3c4d-0000-1111-2222-333344445555"
    assert bench.nvsmi_id(p, 3) == "GPU-1a2b3c4d-0000-1111-2222-333344445555"
    p.uuid = "GPU-1a2b"
    assert bench.nvsmi_id(p, 0) == "GPU-1a2b"


def test_clock_samples_and_phases(bench):
    """nvidia-smi lines parse into (time, SM MHz, max MHz, active reasons);
    phases select the samples between their marks; the line's record counts
    the samples of the timed steps and of the window after them."""
    import datetime
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 250000)
    lines = []
    for i, (mhz, cap) in enumerate([(2070, "Not Active"), (1980, "Active"), (1900, "Not Active")]):
        ts = (t0 + datetime.timedelta(milliseconds=100 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, {mhz}, 2070, 800.5, 0x0, Not Active, Not Active, Not Active, {cap}")
    parsed = [bench.parse_clock_line(x) for x in lines]
    assert all(parsed)
    assert parsed[1][1] == 1980.0 and parsed[1][2] == 2070.0 and parsed[1][3] == {"sw_power_cap"}
    assert abs(parsed[2][0] - parsed[0][0] - 0.2) < 1e-6
    assert bench.parse_clock_line("garbage") is None
    assert bench.parse_clock_line("[N/A], 1, 2, 3, 4, 5, 6, 7, 8") is None
    st = bench.clock_stats(parsed)
    assert st == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                  "samples": 3}
    assert bench.clock_stats([])["samples"] == 0
    rec = bench.line_clocks({"load": st, "timed": bench.clock_stats(parsed[:1])}, 1.0)
    assert rec["samples"] == 3 and rec["samples_in_timed_region"] == 1 and rec["window_s"] == 1.0
    assert bench.line_clocks({}, 1.0) is None


def test_configs_summary(bench):
    """The compact per-configuration record that ends the JSON line: the
    method's configurations only, six numbers each."""
    from residual_add_rmsnorm_gb300 import workloads as W
    pc = {w.name: {"us_per_launch": 10.0, "gbs": 6400.0, "floor_us": 2.0, "sm_mhz": 2070.0}
          for w in W.CONFIGS}
    pc["something_else"] = {"us_per_launch": 1.0, "gbs": 1.0}
    s = bench.configs_summary(pc, 6684.5)
    assert set(s) == {"fields"} | {w.name for w in W.CONFIGS}
    assert s["fused_bf16_T4096_H4096"] == [10.0, 6400.0, round(6400 / 6684.5, 3), 0.8, 2.0,
                                           2070.0]
    assert len(json.dumps(s)) < 1200   # fits the tail of the output with room to spare


def test_plan_fields(bench):
    p = "rows.cta vec16 per_thread=8 block=256 grid=64 cluster=1 smem=0"
    assert bench.plan_field(p, "grid") == 64 and bench.plan_field(p, "block") == 256
    assert bench.plan_field(p, "stages") is None
