"""Host logic of bench.py that needs no GPU: the roofline's measured traffic
is reported only while the recorded ncu figure was taken on the kernel
sources as they stand, for the same workload and row count."""
import json
import os

import bench
from gated_deltanet_layer_gb300 import workloads as WL


def _fake_root(tmp_path):
    for d in ("include", "profiles"):
        (tmp_path / d).mkdir()
    src = tmp_path / "gated_deltanet_layer_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("__global__ void k() {}\n")
    (tmp_path / "include" / "h.h").write_text("/* api */\n")
    return tmp_path


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.kernel_source_hash()
    rec = {"source_sha": sha, "workload": "shard", "rows": 16, "dram_bytes_per_launch": 12345}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.measured_traffic("shard", 16) == 12345
    assert bench.measured_traffic("shard", 8) is None
    assert bench.measured_traffic("full", 16) is None
    # any change to a kernel source or the header makes the record stale
    (root / "gated_deltanet_layer_gb300" / "csrc" / "k.cu").write_text("__global__ void k() { }\n")
    assert bench.kernel_source_hash() != sha
    assert bench.measured_traffic("shard", 16) is None


def test_missing_or_broken_record_gives_no_traffic(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("shard", 16) is None
    (root / "profiles" / "traffic.json").write_text("{not json")
    assert bench.measured_traffic("shard", 16) is None


def test_committed_record_is_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert set(rec) >= {"source_sha", "workload", "rows", "dram_bytes_per_launch"}
    shape = WL.SHAPES[rec["workload"]]
    # DRAM bytes of a launch: at least the weights, at most every counted byte
    # read and written with generous slack for partial-buffer traffic
    assert shape.weight_bytes() <= rec["dram_bytes_per_launch"] <= 1.5 * shape.launch_bytes(rec["rows"])
