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


@pytest.mark.parametrize("code", [0, 1])
@pytest.mark.parametrize("B", [128, 512])
def test_decompress_exact_inputs_see_the_rescaling(B, code):
    """tests/test_gpu_decompress_exact.py: without the 2^64 rescaling, the
    blocks whose factor is subnormal in binary32 (a few bits left) decode to
    other bf16 values than the expected ones.  (The order in which an
    ordinary factor is formed is not resolved there: two orders differ by a
    binary32 ulp, which moves a bf16 output only near a bf16 rounding
    boundary.  With INT8 codes, or E4M3 codes at B = 32, the products of such
    factors are mostly below the bf16 range.)"""
    import oracle
    import test_gpu_decompress_exact as decompress_exact
    _, codes, alpha, s = decompress_exact.crafted_records(B, code, seed=100 * B + 10 * code)
    want = decompress_exact.expected_bits(codes, alpha, s, B, code, rotate=True)
    rB = np.float32(1.0 / np.sqrt(B))
    y = (decode_table(code)[codes] @ hadamard(B).T).astype(np.float32)
    with np.errstate(under="ignore"):
        f = ((s * rB).astype(np.float32) / alpha).astype(np.float32)
        plain = oracle.bf16_round((y * f[:, None]).astype(np.float32).reshape(-1)).reshape(want.shape)
    subnormal = (f > 0) & (f < np.float32(2.0 ** -126))
    assert subnormal.sum() >= 20
    assert np.sum(plain[subnormal] != want[subnormal]) >= 20
