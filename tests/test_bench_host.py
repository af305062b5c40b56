"""bench.py's host-side rules, checked without a GPU: the DRAM traffic a line
reports is the recorded capture's only while the kernel's source is the one that
was captured, and every workload reports its own metric and unit."""
import hashlib
import json
import os

import bench


def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def test_recorded_traffic_is_reported_only_for_the_captured_source():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, e in d.items():
        fresh = _sha(os.path.join(bench.ROOT, e["source"])) == e["sha256"]
        want = int(e["dram_bytes_per_launch"]) * int(e.get("launches_per_call", 1)) if fresh else None
        assert bench.traffic(key) == want, key
    assert bench.traffic(None) is None and bench.traffic("no such kernel") is None


def test_editing_a_captured_source_withdraws_its_traffic(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// the captured source\n")
    (tmp_path / "profiles").mkdir()
    entry = {"kernel": "k", "source": "kernel.cu", "sha256": _sha(src), "dram_bytes_per_launch": 100,
             "launches_per_call": 3}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k/n1": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic("k/n1") == 300
    src.write_text("// the captured source, edited\n")
    assert bench.traffic("k/n1") is None
    src.unlink()
    assert bench.traffic("k/n1") is None


def test_every_workload_reports_its_own_metric_and_unit():
    for name in bench.WORKLOADS:
        metric, unit = bench.metric_for(name), bench.unit_for(name)
        if name.startswith("river"):
            assert metric == bench.RIVER_METRIC and unit == "tokens/s"
        elif name.startswith("ridge"):
            assert metric == bench.RIDGE_METRIC and unit == "rows/s"
        else:
            assert metric == bench.METRIC and unit == "tokens/s"
