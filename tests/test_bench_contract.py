"""bench.py's contract, checked on the host (no GPU): the reference arm's JSON
line and the sha-gated traffic table that feeds roofline.traffic."""
import hashlib
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-rows", "4"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert "workload" in d["config"] and "model" not in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_table_is_used_only_for_the_profiled_source(tmp_path):
    table = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for e in table["entries"]:
        # every record names an existing source file and a whole byte count
        assert os.path.exists(os.path.join(ROOT, e["source"]))
        assert isinstance(e["bytes_per_launch"], int) and e["bytes_per_launch"] > 0
        assert e["command"].count("ncu") >= 1 and "--clock-control none" in e["command"]
    e = table["entries"][0]
    src = os.path.join(ROOT, e["source"])
    # A record is used only while its sha256 prefix matches the source: the
    # kernel source as profiled gives the bytes, a changed copy gives None.
    same = tmp_path / "same.cuh"
    same.write_bytes(open(src, "rb").read())
    changed = tmp_path / "changed.cuh"
    changed.write_bytes(open(src, "rb").read() + b"\n// changed\n")
    sha = hashlib.sha256(same.read_bytes()).hexdigest()[:16]
    for path, expect in ((same, e["bytes_per_launch"]), (changed, None)):
        t = tmp_path / "t.json"
        t.write_text(json.dumps({"entries": [dict(e, source=str(path), source_sha256_16=sha)]}))
        assert bench.traffic_from_profiles(e["kernel"], e["workload"], str(t)) == expect
    assert bench.traffic_from_profiles("no such kernel", e["workload"]) is None
