"""The two exact-arithmetic GPU tests would see the mistake they are for.

tests/test_gpu_compress_exact.py and tests/test_gpu_reduce_exact_sum.py
compare the kernels with binary32 arithmetic formed on the host.  The
plausible mistake both guard against is a product fused into the following
add (the compiler's contraction of a packed multiply and add): the INT8
rounding add then rounds the exact product y * k instead of its binary32
value, and the shard sum adds q * f unrounded.  On the tests' own inputs (no
GPU needed) that mistake must change the expected outputs: INT8 codes of the
compress test, and max|W| (hence s') of the reduce test."""
import numpy as np
import pytest

from helpers import decode_table, hadamard, records
import test_gpu_compress_exact as compress_exact
import test_gpu_reduce_exact_sum as reduce_exact


@pytest.mark.parametrize("B", [32, 128, 512])
@pytest.mark.parametrize("variant", [0, 1])
def test_compress_exact_inputs_separate_rounded_from_fused_int8(B, variant):
    code = 2
    X = compress_exact.integer_blocks(B, seed=100 * B + 10 * code + variant)
    y64 = X.astype(np.float64) @ hadamard(B).T
    y = y64.astype(np.float32)
    ymax = np.abs(y).max(axis=1)
    ordinary = ymax >= np.float32(2.0 ** -100)           # the rescaled blocks take another k
    k = (np.float32(127) / ymax[ordinary]).astype(np.float32)
    u32 = (y[ordinary] * k[:, None]).astype(np.float32)
    fused = np.rint(y64[ordinary] * k[:, None].astype(np.float64))
    assert np.sum(np.rint(u32) != fused) >= 10


@pytest.mark.parametrize("B", [32, 128, 512])
@pytest.mark.parametrize("P", [2, 8, 16])
def test_reduce_exact_inputs_separate_rounded_from_fused_sum(B, P):
    code = 0
    shards, _ = reduce_exact.crafted_shards(P, B, code, seed=1000 * B + 10 * P + code)
    W = reduce_exact.float32_sum(shards, B, code)
    table = decode_table(code)
    fused = np.zeros(W.shape, np.float64)
    for sh in shards:
        c, _, s = records(sh, B)
        fused = (fused + table[c] * s[:, None]).astype(np.float32).astype(np.float64)   # one rounding per add
    changed = np.abs(W).max(axis=1) != np.abs(fused).max(axis=1).astype(np.float32)
    assert changed.sum() >= 50
