"""The benchmark's output line: one JSON object with every key the run
contract names, with sane types and values, measured on the tiny fp32
workload (a few seconds, CPU baseline included)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_carries_the_contract_keys():
    j = run_bench("--workload", "tiny_f32", "--steps", "5", "--warmup", "3")
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("roofline", dict), ("e2e", dict),
                     ("gpu_launches", int), ("clocks", dict), ("cpu_baseline", dict)):
        assert isinstance(j[key], typ), key
    assert "vs_baseline" in j and j["vs_baseline"] is None
    assert j["n_gpus"] == 1 and j["steps"] == 5 and j["warmup"] == 3 and j["scaling"] == "weak"
    assert j["value"] > 0 and j["ms_per_step"] > 0 and j["higher_is_better"] is True
    assert j["config"]["workload"] == "tiny_f32" and j["dtype"] == "f32" and j["data"] == "synthetic"
    r = j["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3 and "traffic" in r
    e = j["e2e"]
    assert e["value"] > 0 and e["unit"] == j["unit"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert j["gpu_launches"] == j["steps"] * 2          # cache write + decode (one partition: no merge)
    c = j["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    b = j["cpu_baseline"]
    assert b["kind"] == "oracle" and b["cores"] >= 1 and b["value"] > 0 and b["unit"] == j["unit"] and b["sample"]
