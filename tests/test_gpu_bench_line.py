"""bench.py on a GB300 keeps its JSON contract: one line with the metric, the
value as defined (2 x 2N bytes of bf16 input over the summed compress and
decompress launch times), the step, roofline, e2e, cpu_baseline, clocks and
parity keys, and a parity block that meets the bar.  Runs the small
[4096 x 1024] workload so that it takes seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "small_4096x1024",
                        "--steps", "40", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
              "step", "ops", "parity"):
        assert k in d, k
    assert d["steps"] == 40 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["gpu_launches"] == 3 * 40
    n = d["config"]["rows"] * d["config"]["hidden"]
    ops = d["ops"]
    want = 4.0 * n / ((ops["compress"]["ms"] + ops["decompress"]["ms"]) * 1e-3) / 1e9
    assert abs(d["value"] - want) <= 1e-9 * want
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-12
    assert d["e2e"]["h2d_bytes_per_step"] == 2 * n and d["e2e"]["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    p = d["parity"]
    for op in ("compress", "reduce"):
        assert p[op]["code_mismatches"] <= p[op]["mismatch_budget"], p
        assert p[op]["code_max_step"] <= 1 and p[op]["alpha_max_rel"] <= 1e-6 and p[op]["s_max_rel"] <= 1e-6, p
    assert p["decompress"]["beyond_one_step"] == 0
    assert d["device_fault_flags"] == 0
