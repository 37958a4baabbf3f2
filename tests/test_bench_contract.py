"""bench.py's reference arm (the CPU oracle on the host cores) keeps the JSON
contract: one line with the metric, value, unit, step counts, config,
cpu_baseline and e2e keys; under a multi-rank launch only rank 0 prints.
Runs on CPU with the small workload, so it takes seconds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "small_4096x1024"]


def run(env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *ARGS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "small_4096x1024"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["cpu_model"] and cb["compiler"].startswith("gcc -O2")
    # The metric: 2 x 2n bytes of bf16 input over the compress + decompress time.
    n = d["config"]["sample_rows"] * d["config"]["hidden"]
    ops = d["ops_ms"]
    assert abs(d["value"] - 4.0 * n / ((ops["compress"] + ops["decompress"]) * 1e-3) / 1e9) <= 1e-9 * d["value"]
    assert abs(d["ms_per_step"] - sum(ops.values())) <= 1e-9 * d["ms_per_step"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("rank", ["1", "3"])
def test_reference_arm_other_ranks_exit_without_work(rank):
    assert run({"RANK": rank, "WORLD_SIZE": "4", "LOCAL_RANK": rank}) == []


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 31, 32, 33, 40, 100, 10000])
@pytest.mark.parametrize("R", [1, 4, 5, 19, 40])
def test_graph_plan_times_exactly_k_steps(K, R):
    """The step graphs cover exactly K steps (K // C replays of C steps plus
    one graph of K mod C), every set-rotating graph is a whole number of
    passes over the R sets, and the per-kernel graphs hold at least the
    minimum number of launches."""
    import bench
    M, L, C = bench.graph_plan(K, R)
    assert L == M * R and L >= bench.LAUNCHES_PER_GRAPH and L - R < bench.LAUNCHES_PER_GRAPH
    assert C % R == 0 and R <= C <= L
    assert (K // C) * C + K % C == K
    if K >= L:
        assert C == L                     # the full graph length once there are enough steps


def test_graph_plan_rejects_empty_runs():
    import bench
    with pytest.raises(ValueError):
        bench.graph_plan(0, 4)
