"""The seeded input generator: determinism, independence of row ranges, and
the shape of each distribution (what the workloads say they draw)."""
import numpy as np

import workloads
from helpers import bf16_to_f64


def test_row_ranges_are_independent_and_deterministic():
    a = workloads.generate("student_t_channels", 64, 512, seed=3)
    b = workloads.generate("student_t_channels", 64, 512, seed=3, row_start=10, row_count=5)
    c = workloads.generate_rows("student_t_channels", 512, 3, [10, 11, 12, 13, 14])
    assert np.array_equal(a[10:15], b) and np.array_equal(b, c)
    t = workloads.generate("student_t_channels", 64, 512, seed=3, threads=4)
    assert np.array_equal(a, t)
    assert not np.array_equal(a, workloads.generate("student_t_channels", 64, 512, seed=4))


def test_uniform_is_inside_open_interval():
    u = np.array([workloads.uniform(0, 0, i) for i in range(20000)])
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01


def test_laplace_outliers_shape():
    x = bf16_to_f64(workloads.generate("laplace_outliers", 512, 4096, seed=0))
    out = np.abs(x) >= 0.05
    assert 0.0007 < out.mean() < 0.0013                   # 0.1% outliers (+ a tiny Laplace tail)
    bulk = x[~out]
    assert abs(np.abs(bulk).mean() / 1e-3 - 1) < 0.02      # E|x| = b for Laplace(0, b)
    assert np.abs(x).max() <= 0.5                          # U[0.05, 0.5) after bf16 rounding


def test_gaussian_sparse_shape():
    x = bf16_to_f64(workloads.generate("gaussian_sparse", 256, 5120, seed=0))
    assert abs((x == 0).mean() - 0.2) < 0.005             # 20% exact zeros
    nz = x[x != 0]
    assert abs(np.median(np.abs(nz)) / (0.6745 * 1e-5) - 1) < 0.02   # sd 1e-5 bulk (median |z| = 0.6745 sd)
    assert 3e-4 < (np.abs(x) > 1e-3).mean() < 5e-4         # 0.05% x1000 (of the 80% non-zero)


def test_student_t_channels_have_column_scales():
    x = bf16_to_f64(workloads.generate("student_t_channels", 2048, 512, seed=0))
    col = np.median(np.abs(x), axis=0)
    ratio = col.max() / col.min()
    assert 10 < ratio < 40                                 # multipliers span [0.25, 8)
    assert np.all(np.isfinite(x))


def test_workload_table():
    w = workloads.WORKLOADS
    assert w["gpt_activation_8192x4096"].numel == 8192 * 4096
    assert w["large_16384x8192"].blocks == (64, 128, 256)
    assert w["shard_reduce_p8_8192x5120"].seeds == tuple(range(8))
