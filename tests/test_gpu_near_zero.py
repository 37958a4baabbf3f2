"""GPU parity in the near-zero region (TACO paper, Section 4.2.1 and Fig. 5:
the Adaptive Scale exists for blocks whose values crowd towards zero;
Section 4.3, Eqs. 9-10: the Dual-Scale step divides by the block maximum).

The blocks of tests/near_zero.py sit at the bottom of the binary32 / bf16
range: x = c (e_0 + e_1) with c = 2^-120 and 2^-125, bf16 subnormals down to
2^-133, and blocks whose max|H G| lies just below and just above
Q_max / FLT_MAX, where Q_max / max|H G| first overflows binary32.  The oracle
scales by alpha ~ 1e15 before it rotates, so none of its values are tiny; the
kernels work on the unscaled rotation and must give the same records.

Every block size (32 .. 512) and both FP8 formats, through compress (against
the oracle's records, element by element), decompress (the GPU decodes the
oracle's records) and the shard reduce (the GPU reduces the oracle's shards).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import bf16_to_f64, records
from near_zero import CODE_QMAX, near_zero_blocks
from parity import compare_decoded, compare_records, exact_compress_u, exact_reduce_scales, reduce_exact_u

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BLOCKS = [32, 64, 128, 256, 512]
CODES = [0, 1]


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def from_dev(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


def no_nan_codes(codes, code):
    c7 = np.asarray(codes) & 0x7F
    return not np.any(c7 == 0x7F) if code == 0 else not np.any(c7 > 0x7B)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", BLOCKS)
def test_near_zero_compress(taco, B, code):
    X = near_zero_blocks(B, code)
    nb = X.shape[0]
    ref = oracle.compress(X.reshape(-1), B, 0, code)
    got = taco.compress(to_dev(X), B, code=code).cpu().numpy()
    cg, ag, sg = records(got, B)
    assert no_nan_codes(cg, code)
    stats = compare_records(got, ref, B, code=code, u_exact=exact_compress_u(X, B, 0, code))
    assert stats["code_mismatches"] == 0, stats
    # Every block is nonzero: its largest code is +-Q_max (Eqs. 9-10).
    top = 0x7E if code == 0 else 0x7B
    assert np.all(np.max(cg & 0x7F, axis=1) == top)
    assert np.all(sg > 0) and nb == cg.shape[0]
    assert taco.device_status() == 0


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", BLOCKS)
def test_near_zero_decompress(taco, B, code):
    X = near_zero_blocks(B, code)
    nb = X.shape[0]
    ref = oracle.compress(X.reshape(-1), B, 0, code)
    y = from_dev(taco.decompress(torch.from_numpy(ref).to(DEV), nb, B, B, code=code))
    y_ref = oracle.decompress(ref, X.size, B, 0, code)
    compare_decoded(y, y_ref, B)
    # The first blocks are exact: c (e_0 + e_1) and single elements come back bit for bit.
    for r in (0, 1, 2, 3):
        assert np.array_equal(y.reshape(nb, B)[r], y_ref.reshape(nb, B)[r]), r
    assert taco.device_status() == 0


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", BLOCKS)
def test_near_zero_reduce(taco, B, code):
    X = near_zero_blocks(B, code)
    nb = X.shape[0]
    n = X.size
    a = oracle.compress(X.reshape(-1), B, 0, code)
    b = oracle.compress(near_zero_blocks(B, code, seed=99).reshape(-1), B, 0, code)
    neg = oracle.compress(X.reshape(-1) ^ np.uint16(0x8000), B, 0, code)
    # A shard of ordinary magnitude next to a tiny one: the sum is the ordinary one.
    big = oracle.compress(workloads.generate("laplace_outliers", nb, B, 5).reshape(-1), B, 0, code)
    for shards in ([a], [a, b], [a, a, a], [b, a, b, a, b], [big, a], [a, neg]):
        ref = oracle.reduce_shards(shards, n, B, 0, code)
        got = taco.reduce_shards([torch.from_numpy(s).to(DEV) for s in shards], nb, B, B, code=code).cpu().numpy()
        cg, _, sg = records(got, B)
        assert no_nan_codes(cg, code)
        compare_records(got, ref, B, code=code, u_exact=reduce_exact_u(shards, B, 0, code),
                        scales_exact=exact_reduce_scales(shards, B, 0, code))
    # A shard and its negation cancel to the all-zero record.
    assert np.all(cg == 0) and np.all(sg == 0)
    assert taco.device_status() == 0


@pytest.mark.parametrize("B", BLOCKS)
def test_near_zero_round_trip_is_exact_on_grid_inputs(taco, B):
    """c (56 h_i + 28 h_j) lands on the E4M3 grid (codes +-448, +-224, 0), so
    decompress(compress(x)) == x bit for bit, here with c so small that the
    inputs are bf16 subnormals or near the bottom of the normal range."""
    from helpers import hadamard
    H = hadamard(B)
    rows = []
    for c, (i, j) in ((2.0 ** -133, (0, 1)), (2.0 ** -131, (3, B - 1)), (2.0 ** -126, (B // 2, 5))):
        rows.append(c * (56 * H[i] + 28 * H[j]))
    X = np.stack([oracle.bf16_round(np.asarray(r, dtype=np.float32)) for r in rows])
    assert np.array_equal(bf16_to_f64(X), np.stack(rows))       # exact in bf16
    packed = taco.compress(to_dev(X), B)
    y = from_dev(taco.decompress(packed, X.shape[0], B, B))
    assert np.array_equal(y, X.reshape(-1))
    got, ref = packed.cpu().numpy(), oracle.compress(X.reshape(-1), B)
    compare_records(got, ref, B)
    assert np.array_equal(records(got, B)[0], records(ref, B)[0])
