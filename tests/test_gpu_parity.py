"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs: element by element at sizes that span many warp tiles
with ragged and odd tails, for every supported block size and distribution,
plus the operator's special cases.  Tolerances are in tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import hadamard, records
from parity import (RELL2_ATOL, compare_decoded, compare_records, exact_reduce_scales, oracle_compress_parallel,
                    oracle_decompress_parallel, reduce_exact_u, rel_l2_bf16)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def to_dev(x_bits: np.ndarray, shape=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16)
    if shape is not None:
        t = t.reshape(shape)
    return t.to(DEV)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


def u8_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# (rows, hidden, block): many tiles, ragged last tile, odd block counts.
SHAPES = [
    (333, 128, 128),      # 333 blocks: odd, last tile of 13
    (517, 256, 128),      # 1034 blocks
    (1001, 64, 64),       # 1001 blocks: odd
    (640, 320, 64),       # 3200 blocks
    (31, 256, 256),       # 31 blocks: odd, last 16-block tile of 15
    (257, 512, 256),      # 514 blocks
    (4096, 1024, 128),    # the small workload itself: every warp loops several times
]
DISTS = ["laplace_outliers", "student_t_channels", "gaussian_sparse"]


@pytest.mark.parametrize("rows,hidden,block", SHAPES)
@pytest.mark.parametrize("dist", DISTS)
def test_compress_decompress_parity(taco, rows, hidden, block, dist):
    x = workloads.generate(dist, rows, hidden, seed=11).reshape(-1)
    ref = oracle_compress_parallel(x, block)
    xd = to_dev(x, (rows, hidden))
    packed = taco.compress(xd, block)
    torch.cuda.synchronize()
    got = packed.cpu().numpy()
    compare_records(got, ref, block)

    # Decompress in isolation: the GPU decodes the ORACLE's records.
    y_gpu = bits_of(taco.decompress(u8_dev(ref), rows, hidden, block))
    y_ref = oracle_decompress_parallel(ref, x.size, block)
    compare_decoded(y_gpu, y_ref, block)

    # Round trip on the GPU vs the oracle's round trip.
    y_rt = bits_of(taco.decompress(packed, rows, hidden, block))
    assert abs(rel_l2_bf16(y_rt, x) - rel_l2_bf16(y_ref, x)) <= RELL2_ATOL
    assert taco.device_status() == 0


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16])
def test_reduce_parity(taco, block, P):
    """GPU reduce of the oracle's packed shards against the oracle's reduce.
    With two shards, exact rounding ties are common (u' = Q_max (q1 f1 + q2 f2) /
    max|W| is an exact E4M3 midpoint whenever the shards' codes share a ratio
    such as 3/4 at an element and at the block maximum); a one-step difference
    at such a tie is an FP32 rounding-order effect and is counted separately."""
    rows, hidden = 797, 2 * block         # 1594 blocks
    xs = [workloads.generate("student_t_channels", rows, hidden, seed=p).reshape(-1) for p in range(P)]
    packed = [oracle.compress(x, block) for x in xs]
    ref = oracle.reduce_shards(packed, xs[0].size, block)
    got = taco.reduce_shards([u8_dev(p) for p in packed], rows, hidden, block)
    torch.cuda.synchronize()
    compare_records(got.cpu().numpy(), ref, block, u_exact=reduce_exact_u(packed, block),
                    scales_exact=exact_reduce_scales(packed, block))


@pytest.mark.parametrize("block", [32, 512])
@pytest.mark.parametrize("P", [2, 4, 16])
def test_reduce_parity_fixed_shard_counts(taco, block, P):
    """The 2-, 4- and 16-shard kernels (tiles of 4x, 2x and 1/2x the usual
    length) at the smallest and largest block, on a shape whose last tile is
    partial and has an odd number of blocks."""
    rows, hidden = 301, 3 * block          # 903 blocks
    xs = [workloads.generate("student_t_channels", rows, hidden, seed=20 + p).reshape(-1) for p in range(P)]
    packed = [oracle.compress(x, block) for x in xs]
    ref = oracle.reduce_shards(packed, xs[0].size, block)
    got = taco.reduce_shards([u8_dev(p) for p in packed], rows, hidden, block)
    torch.cuda.synchronize()
    compare_records(got.cpu().numpy(), ref, block, u_exact=reduce_exact_u(packed, block),
                    scales_exact=exact_reduce_scales(packed, block))
    assert taco.device_status() == 0


def test_reduce_repeated_and_negated_shards(taco):
    block, rows, hidden = 128, 64, 512
    x = workloads.generate("laplace_outliers", rows, hidden, seed=3).reshape(-1)
    p = oracle.compress(x, block)
    neg = oracle.compress(x ^ np.uint16(0x8000), block)
    pd, nd = u8_dev(p), u8_dev(neg)
    # Same shard twice (aliasing inputs is allowed).
    got = taco.reduce_shards([pd, pd, pd], rows, hidden, block).cpu().numpy()
    compare_records(got, oracle.reduce_shards([p, p, p], x.size, block), block)
    # A shard and its negation cancel exactly: the all-zero record.
    z = taco.reduce_shards([pd, nd], rows, hidden, block).cpu().numpy()
    c, a, s = records(z, block)
    assert np.all(c == 0) and np.all(s == 0)
    assert np.all(a == np.float32(1.0) / np.sqrt(np.float32(1e-30)))


@pytest.mark.parametrize("block", [64, 128, 256])
def test_special_blocks(taco, block):
    B = block
    H = hadamard(B)
    rows = []
    rows.append(np.zeros(B))                                   # all-zero block
    rows.append(np.full(B, 0.75))                              # constant block
    rows.append(np.full(B, -2.0 ** 40))                        # large constant
    one = np.zeros(B); one[5] = -3.0; rows.append(one)         # single nonzero element
    rows.append(1e-30 * H[3])                                  # tiny values
    negz = np.zeros(B); rows.append(-negz)                     # negative zeros
    a, b = 56, 28
    for i, j in [(0, 1), (7, B - 1), (B // 2, 3)]:
        rows.append(2.0 ** -7 * (a * H[i] + b * H[j]))        # lands on the E4M3 grid
    X = np.array(rows, dtype=np.float32)
    x = oracle.bf16_round(X)
    if len(rows) > 0:
        x = x.copy()
        x[5 * B:6 * B] = 0x8000                                # -0.0 in bf16
    ref = oracle.compress(x, B)
    got = taco.compress(to_dev(x, (len(rows), B)), B).cpu().numpy()
    compare_records(got, ref, B)
    cg, ag, sg = records(got, B)
    assert np.all(cg[0] == 0) and sg[0] == 0                   # all-zero rule
    assert np.all(cg[5] == 0) and sg[5] == 0                   # negative zeros: codes 0x00
    assert cg[1, 0] == 0x7E and np.all((cg[1, 1:] & 0x7F) == 0)
    assert cg[2, 0] == 0xFE and np.all((cg[2, 1:] & 0x7F) == 0)
    assert set(np.unique(cg[3])) <= {0x7E, 0xFE}
    # Grid inputs come back bit-exactly; zero blocks come back as +0.
    y = bits_of(taco.decompress(u8_dev(got), len(rows), B, B)).reshape(len(rows), B)
    assert np.all(y[0] == 0) and np.all(y[5] == 0)
    for r in (1, 2, 6, 7, 8):
        assert np.array_equal(y[r], x.reshape(len(rows), B)[r]), r


def test_empty_tensor_is_a_no_op(taco):
    lib = taco.load_library()
    assert lib.taco_compress(None, 0, 128, 128, None, None) == 0
    assert lib.taco_decompress(None, 5, 0, 64, None, None) == 0
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    assert taco.compress(x, 128).numel() == 0
    assert taco.decompress(torch.empty(0, dtype=torch.uint8, device=DEV), 0, 256, 128).numel() == 0


def test_argument_errors_launch_nothing(taco):
    lib = taco.load_library()
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device=DEV)
    out = torch.full((taco.compressed_bytes(16, 256, 128) + 64,), 7, dtype=torch.uint8, device=DEV)
    xp, op = x.data_ptr(), out.data_ptr()
    assert lib.taco_compress(xp, 16, 256, 96, op, None) == 3          # unsupported block
    assert lib.taco_compress(xp, 16, 200, 128, op, None) == 2         # hidden % block
    assert lib.taco_compress(xp, -1, 256, 128, op, None) == 2         # negative rows
    assert lib.taco_compress(None, 16, 256, 128, op, None) == 1       # null input
    assert lib.taco_compress(xp + 2, 16, 256, 128, op, None) == 4     # misaligned input
    assert lib.taco_compress(xp, 16, 256, 128, op + 8, None) == 4     # misaligned output
    assert lib.taco_compress(xp, 16, 256, 128, xp + 16, None) == 6    # output overlaps input
    assert lib.taco_decompress(op, 16, 256, 128, op + 1024, None) in (4, 6)
    ptrs = (taco._binding.ctypes.c_void_p * 17)(*([op] * 17))
    assert lib.taco_reduce_shards(ptrs, 0, 16, 256, 128, xp, None) == 5
    assert lib.taco_reduce_shards(ptrs, 17, 16, 256, 128, xp, None) == 5
    assert lib.taco_reduce_shards(ptrs, 2, 16, 256, 128, op, None) == 6   # out overlaps a shard
    torch.cuda.synchronize()
    assert torch.all(out == 7)                                           # untouched
    with pytest.raises(taco.TacoError):
        taco.compress(x, 96)
    assert lib.taco_abi_version() == 2


def test_streams_are_respected(taco):
    """Work goes on the caller's stream: results are complete after that
    stream (not the default one) is synchronised."""
    rows, hidden, block = 2048, 1024, 128
    x = workloads.generate("laplace_outliers", rows, hidden, seed=5).reshape(-1)
    xd = to_dev(x, (rows, hidden))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        packed = taco.compress(xd, block, stream=s)
        y = taco.decompress(packed, rows, hidden, block, stream=s)
    s.synchronize()
    ref = oracle_compress_parallel(x, block)
    compare_records(packed.cpu().numpy(), ref, block)
    assert taco.device_status(stream=s) == 0
    assert abs(rel_l2_bf16(bits_of(y), x) - rel_l2_bf16(oracle_decompress_parallel(ref, x.size, block), x)) < 1e-6
