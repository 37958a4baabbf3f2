"""GPU parity of the ablation variants and code formats (the _ex calls)
against the CPU oracle on the same seeded inputs.

Variants (paper Sections 5.2.2, 5.3.1): ASH + DS, standard Hadamard + DS,
DS only, ASH only.  Codes (Section 5.3.2; Sections 2 and 6): E4M3, E5M2,
INT8.  Same bar as the method itself: scales to 1e-6 relative, codes
identical except at most 1e-4 of the elements and those one grid step apart
(rounding ties of the exact value counted apart), decoded bf16 within one
step where FP32 noise reaches a midpoint, reconstruction RelL2 within 1e-3
of the oracle's.  Every CUDA input that stands in for a received record
comes from the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import bf16_to_f64, records
from parity import (RELL2_ATOL, compare_decoded, compare_records, exact_compress_u, exact_reduce_scales,
                    oracle_compress_parallel,
                    oracle_decompress_parallel, reduce_exact_u, rel_l2_bf16)

pytestmark = pytest.mark.gpu

VARIANTS = [0, 1, 2, 3]
CODES = [0, 1, 2]
ROWS, HIDDEN = 300, 1024     # 2400 blocks at B = 128: 18.75 compress tiles, ragged


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def from_dev(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


BLOCKS = [32, 64, 128, 256, 512]


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("B", BLOCKS)
def test_compress_decompress(taco, B, variant, code):
    bits = workloads.generate("laplace_outliers", ROWS, HIDDEN, 11 + variant + 4 * code)
    n = bits.size
    ref = oracle_compress_parallel(bits, B, variant, code)
    got = taco.compress(to_dev(bits).view(ROWS, HIDDEN), B, variant=variant, code=code).cpu().numpy()
    u = exact_compress_u(bits, B, variant, code)
    compare_records(got, ref, B, u_exact=u, code=code)
    # Decompress the oracle's records on the GPU.
    y = from_dev(taco.decompress(torch.from_numpy(ref).cuda(), ROWS, HIDDEN, B, variant=variant, code=code))
    y_ref = oracle_decompress_parallel(ref, n, B, variant, code)
    compare_decoded(y, y_ref, B)
    # Whole round trip on the GPU against the oracle's.
    y_gpu = from_dev(taco.decompress(torch.from_numpy(got).cuda(), ROWS, HIDDEN, B, variant=variant, code=code))
    assert abs(rel_l2_bf16(y_gpu, bits) - rel_l2_bf16(y_ref, bits)) <= RELL2_ATOL
    assert taco.device_status() == 0


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("B", BLOCKS)
def test_reduce(taco, B, variant, code):
    rows, hidden, P = 96, 1024, 3
    shards = [oracle.compress(workloads.generate("student_t_channels", rows, hidden, p), B, variant, code)
              for p in range(P)]
    n = rows * hidden
    ref = oracle.reduce_shards(shards, n, B, variant, code)
    got = taco.reduce_shards([torch.from_numpy(s).cuda() for s in shards], rows, hidden, B,
                             variant=variant, code=code).cpu().numpy()
    u = reduce_exact_u(shards, B, variant, code)
    compare_records(got, ref, B, u_exact=u, code=code, scales_exact=exact_reduce_scales(shards, B, variant, code))
    assert taco.device_status() == 0


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", [0, 1, 3])
@pytest.mark.parametrize("B", BLOCKS)
def test_reduce_eight_shards(taco, B, variant, code):
    # Eight shards run the kernels with the shard loop unrolled; odd block
    # counts (B = 512) leave a record outside the tile copies.
    rows, hidden, P = 97, 1536, 8
    shards = [oracle.compress(workloads.generate("student_t_channels", rows, hidden, 40 + p), B, variant, code)
              for p in range(P)]
    n = rows * hidden
    ref = oracle.reduce_shards(shards, n, B, variant, code)
    got = taco.reduce_shards([torch.from_numpy(s).cuda() for s in shards], rows, hidden, B,
                             variant=variant, code=code).cpu().numpy()
    u = reduce_exact_u(shards, B, variant, code)
    compare_records(got, ref, B, u_exact=u, code=code, scales_exact=exact_reduce_scales(shards, B, variant, code))
    assert taco.device_status() == 0


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_special_blocks(taco, variant, code):
    """All-zero, single-spike and constant blocks, and a shard with its
    negation, through every variant and code format."""
    B = 128
    G = np.zeros((6, B))
    G[1, 5] = 3.0
    G[2, :] = -0.25
    G[3, 0] = 1e-3
    G[3, 77] = -2e-3
    G[4] = np.linspace(-1, 1, B)
    G[5, ::3] = 7.5
    bits = oracle.bf16_round(G.astype(np.float32))
    ref = oracle.compress(bits, B, variant, code)
    got = taco.compress(to_dev(bits).view(6, B), B, variant=variant, code=code).cpu().numpy()
    compare_records(got, ref, B, code=code)
    neg = oracle.compress(bits ^ np.uint16(0x8000), B, variant, code)
    r = taco.reduce_shards([torch.from_numpy(ref).cuda(), torch.from_numpy(neg).cuda()], 6, B, B,
                           variant=variant, code=code).cpu().numpy()
    compare_records(r, oracle.reduce_shards([ref, neg], bits.size, B, variant, code), B, code=code)
    c, a, s = records(r, B)
    assert np.all(s == (1.0 if variant == 3 else 0.0))
    assert taco.device_status() == 0


@pytest.mark.parametrize("B", [32, 512])
def test_small_and_large_blocks_ragged(taco, B):
    """Blocks 32 and 512 (the warp-per-block codec) on shapes with an odd
    number of blocks, a partial last tile of the shard reduce and a single
    block, for the method itself."""
    for rows, hidden in ((301, 3 * B), (1, B), (7, 5 * B)):
        bits = workloads.generate("gaussian_sparse", rows, hidden, rows)
        ref = oracle.compress(bits, B)
        got = taco.compress(to_dev(bits).view(rows, hidden), B).cpu().numpy()
        compare_records(got, ref, B)
        y = from_dev(taco.decompress(torch.from_numpy(ref).cuda(), rows, hidden, B))
        compare_decoded(y, oracle.decompress(ref, bits.size, B), B)
        shards = [ref, oracle.compress(workloads.generate("laplace_outliers", rows, hidden, 99), B)]
        r = taco.reduce_shards([torch.from_numpy(x).cuda() for x in shards], rows, hidden, B).cpu().numpy()
        u = reduce_exact_u(shards, B)
        compare_records(r, oracle.reduce_shards(shards, bits.size, B), B, u_exact=u)
    assert taco.device_status() == 0


def test_default_matches_plain_calls(taco):
    """variant 0 / code 0 through the binding is the plain call (same bytes)."""
    bits = workloads.generate("laplace_outliers", 64, 1024, 1)
    x = to_dev(bits).view(64, 1024)
    a = taco.compress(x, 128).cpu().numpy()
    b = taco.compress(x, 128, variant="ash_ds", code="e4m3").cpu().numpy()
    assert np.array_equal(a, b)
