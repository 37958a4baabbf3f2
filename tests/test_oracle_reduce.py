"""Pins of the oracle's shard reduction (the single local reduction of the
two-shot AllReduce, Section 4.4.2): decode P shards, sum in FP32, compress once.

Because (1/sqrt B) H_B is symmetric and orthogonal (Section 4.2.2), the sum of
the decoded shards is S = (1/sqrt B) H W with W = sum_p q_p s_p / alpha_p, so in
real arithmetic the re-compressed codes are u' = Q_max W / max|W| and
s'/alpha' = max|W| / Q_max.  The tests check the oracle against that closed form
and against its special cases:

- P = 1: the codes come back unchanged and s'/alpha' = s/alpha;
- P identical shards: the same codes and P times the ratio;
- a shard and its negation: all-zero blocks (s = 0, codes 0);
- eight workload shards: every code within half an E4M3 step of u'.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import QMAX, TAU, e4m3_decode_table, e4m3_half_ulp, records


def shard_inputs(P, rows=16, hidden=512, dist="student_t_channels"):
    return [workloads.generate(dist, 8192, hidden, seed=p, row_count=rows).reshape(-1) for p in range(P)]


@pytest.mark.parametrize("B", [64, 128, 256])
def test_single_shard_is_idempotent(B):
    x = shard_inputs(1)[0]
    p = oracle.compress(x, B)
    r = oracle.reduce_shards([p], x.size, B)
    c0, a0, s0 = records(p, B)
    c1, a1, s1 = records(r, B)
    t = e4m3_decode_table()
    assert np.array_equal(t[c0], t[c1])
    assert np.all(np.abs((s1 / a1) / (s0 / a0) - 1) < 1e-6)


@pytest.mark.parametrize("P", [2, 3, 8])
def test_identical_shards_scale_the_ratio(P):
    B = 128
    x = shard_inputs(1)[0]
    p = oracle.compress(x, B)
    r = oracle.reduce_shards([p] * P, x.size, B)
    c0, a0, s0 = records(p, B)
    c1, a1, s1 = records(r, B)
    t = e4m3_decode_table()
    assert np.array_equal(t[c0], t[c1])
    assert np.all(np.abs((s1 / a1) / (P * s0 / a0) - 1) < 1e-6)


def test_shard_and_its_negation_cancel():
    B = 128
    x = shard_inputs(1)[0]
    neg = x ^ np.uint16(0x8000)
    p, n = oracle.compress(x, B), oracle.compress(neg, B)
    c, a, s = records(oracle.reduce_shards([p, n], x.size, B), B)
    assert np.all(s == 0)
    assert np.all(c == 0)
    assert np.all(a == np.float32(1.0) / np.sqrt(np.float32(1e-30)))


@pytest.mark.parametrize("B", [64, 128, 256])
def test_eight_shards_against_closed_form(B):
    xs = shard_inputs(8)
    packed = [oracle.compress(x, B) for x in xs]
    out = oracle.reduce_shards(packed, xs[0].size, B)
    t = e4m3_decode_table()
    W = 0
    for p in packed:
        c, a, s = records(p, B)
        W = W + t[c] * (s / a)[:, None]
    wmax = np.abs(W).max(axis=1)
    u = QMAX * W / wmax[:, None]
    c1, a1, s1 = records(out, B)
    q = t[c1]
    assert np.all(np.abs(q - u) <= e4m3_half_ulp(u) + QMAX * 4e-6)
    assert np.all(np.abs((s1 / a1) / (wmax / QMAX) - 1) < 2e-6)
    # The new alpha brings the energy of the sum to the target (Eq. 7):
    # mean(S^2) = |W|^2 / B by orthogonality.
    m = (W ** 2).sum(axis=1) / B
    assert np.all(np.abs(a1 * np.sqrt(m) / TAU - 1) < 1e-6)


def test_reduce_of_decoded_sum_matches_float32_pipeline():
    """reduce_shards equals compress_f32 of the float32 sum of decompress_f32
    (the same definition, spelled out through the oracle's public pieces)."""
    B = 128
    xs = shard_inputs(3)
    packed = [oracle.compress(x, B) for x in xs]
    acc = np.zeros(xs[0].size, dtype=np.float32)
    for p in packed:
        acc = acc + oracle.decompress_f32(p, xs[0].size, B)
    assert np.array_equal(oracle.compress_f32(acc, B), oracle.reduce_shards(packed, xs[0].size, B))
