"""Hand-derived worked examples (tests/golden/worked_examples.json, each with
the equations it follows) and the oracle's regression digests."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from helpers import bf16_to_f64, records

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
    DATA = json.load(f)


def closed_form(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt}))


def bf16(x):
    return oracle.bf16_round(np.asarray(x, dtype=np.float32))


def check_record(packed, ex):
    B = ex["B"]
    codes, alpha, s = records(packed, B)
    assert [f"0x{c:02x}" for c in codes[0]] == ex["codes"]
    a_ref, s_ref = closed_form(ex["alpha"]), closed_form(ex["s"])
    assert abs(alpha[0] / a_ref - 1) < 1e-6
    if s_ref == 0:
        assert s[0] == 0
    else:
        assert abs(s[0] / s_ref - 1) < 1e-6
    out = bf16_to_f64(oracle.decompress(packed, B, B))
    assert np.array_equal(out, np.array(ex["decoded"]))


@pytest.mark.parametrize("ex", DATA["examples"], ids=lambda e: e["name"])
def test_worked_example(ex):
    check_record(oracle.compress(bf16(ex["x"]), ex["B"]), ex)


@pytest.mark.parametrize("ex", DATA["reductions"], ids=lambda e: e["name"])
def test_worked_reduction(ex):
    B = ex["B"]
    shards = [oracle.compress(bf16(x), B) for x in ex["shards"]]
    check_record(oracle.reduce_shards(shards, B, B), ex)


def test_regression_digests():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_regression", os.path.join(GOLDEN, "make_regression.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "regression.txt")) as f:
        stored = f.read().split("\n")
    assert mod.digests() == [l for l in stored if l]
