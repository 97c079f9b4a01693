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
    names = {w.name for w in bench._configs()} | {bench.FP8IN_NAME}
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
