"""Host-side pieces of bench.py that need no GPU: the CPU baseline's report
(all cores and one core), and the rule that DRAM traffic from the committed
ncu summary is reported only while the kernel sources are the ones it was
captured on."""
from __future__ import annotations

import json
import os
import shutil

import pytest

import workloads


def _bench():
    import bench
    return bench


def test_cpu_baseline_reports_all_cores_and_one():
    pytest.importorskip("numpy")
    bench = _bench()
    case = workloads.make_config("tiny_f32")
    r = bench.cpu_baseline(case, 0.3)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s"
    assert r["value"] > 0 and r["cores"] >= 1
    assert r["host_cpus"] == os.cpu_count()
    one = r["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == "tokens/s"
    import oracle
    assert oracle.max_threads() == r["cores"], "the baseline restores the oracle's thread count"


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    bench = _bench()
    committed = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    key = "record:rollback_b128_t16_bf16"
    assert key in committed["kernels"]
    # a copy of the tree's profile with the current hash: the entry is read
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    fresh = dict(committed, kernel_source_hash=bench.kernel_source_hash())
    (root / "profiles" / "traffic.json").write_text(json.dumps(fresh))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("record", "rollback_b128_t16_bf16") == \
        committed["kernels"][key]["dram_bytes_per_launch"]
    assert bench.measured_traffic("record", "no_such_workload") is None
    # any other hash (sources changed since the capture): nothing is reported
    stale = dict(committed, kernel_source_hash="0" * 16)
    (root / "profiles" / "traffic.json").write_text(json.dumps(stale))
    assert bench.measured_traffic("record", "rollback_b128_t16_bf16") is None


def test_kernel_source_hash_follows_the_sources(tmp_path, monkeypatch):
    bench = _bench()
    src = tmp_path / "csrc"
    shutil.copytree(bench.KERNEL_SOURCES, src)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", str(src))
    h0 = bench.kernel_source_hash()
    (src / "notes.txt").write_text("not a source file")
    assert bench.kernel_source_hash() == h0
    cu = sorted(p for p in os.listdir(src) if p.endswith(".cuh"))[0]
    with open(src / cu, "a") as f:
        f.write("\n// edited\n")
    assert bench.kernel_source_hash() != h0
