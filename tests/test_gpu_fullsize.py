"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times (one call over the whole tensor), element by element over the
whole tensor:

- compress: the GPU's records against the oracle's (the oracle runs over the
  whole tensor, block ranges on several host threads);
- decompress: the GPU decodes the oracle's records, and every bf16 output is
  checked against the oracle's decode of the same records;
- the reconstruction relative L2 error of the GPU's own round trip against the
  oracle's;
- the 8-shard reduce: the GPU reduces the oracle's shards, against the
  oracle's reduce of the same shards, and the GPU decodes the oracle's
  reduced records; plus the whole pipeline on the GPU.

A sample of blocks (and both ends) is also recomputed by the oracle one block
at a time, independently of the threaded runs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (RELL2_ATOL, compare_decoded, compare_records, oracle_compress_parallel,
                    oracle_decompress_parallel, oracle_reduce_parallel, reduce_exact_u, rel_l2_bf16,
                    exact_compress_scales, exact_compress_u, exact_reduce_scales)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"
N_SAMPLE = 3000


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def to_dev(x_bits, rows, hidden):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).reshape(
        rows, hidden).to(DEV)


def sample_blocks(nblocks, seed):
    rng = np.random.default_rng(seed)
    s = rng.choice(nblocks, size=min(N_SAMPLE, nblocks), replace=False)
    return np.unique(np.concatenate([s, [0, 1, nblocks - 2, nblocks - 1]]))


def block_rows(packed, ids, block):
    rec = packed.reshape(-1, block + 8)
    return rec[ids].reshape(-1)


CASES = [("small_4096x1024", 128), ("gpt_activation_8192x4096", 128), ("tp_grad_8192x5120", 128),
         ("large_16384x8192", 64), ("large_16384x8192", 128), ("large_16384x8192", 256),
         ("large_16384x8192", 32), ("large_16384x8192", 512)]


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


@pytest.mark.parametrize("name,block", CASES)
def test_full_size_compress_decompress(taco, name, block):
    w = workloads.WORKLOADS[name]
    x = w.tensor().reshape(-1)
    nblocks = x.size // block
    xd = to_dev(x, w.rows, w.hidden)
    packed = taco.compress(xd, block)
    y = taco.decompress(packed, w.rows, w.hidden, block)
    torch.cuda.synchronize()
    assert taco.device_status() == 0
    got = packed.cpu().numpy()
    y_gpu = bits_of(y)
    del xd, packed, y
    # Sampled blocks recomputed one by one.
    ids = sample_blocks(nblocks, 1)
    xs = x.reshape(-1, block)[ids].reshape(-1)
    compare_records(block_rows(got, ids, block), oracle.compress(xs, block), block)
    # Every record of the tensor.
    ref = oracle_compress_parallel(x, block)
    compare_records(got, ref, block, scales_exact=exact_compress_scales(x, block))
    # Decompress in isolation: the GPU decodes the oracle's records, every element checked.
    y_ref = oracle_decompress_parallel(ref, x.size, block)
    y_dec = bits_of(taco.decompress(torch.from_numpy(ref).to(DEV), w.rows, w.hidden, block))
    assert taco.device_status() == 0
    compare_decoded(y_dec, y_ref, block)
    ys = oracle.decompress(block_rows(ref, ids, block), ids.size * block, block)
    assert np.array_equal(y_ref.reshape(-1, block)[ids].reshape(-1), ys)
    # Whole-tensor reconstruction error against the oracle's.
    e_gpu, e_ref = rel_l2_bf16(y_gpu, x), rel_l2_bf16(y_ref, x)
    assert abs(e_gpu - e_ref) <= RELL2_ATOL, (e_gpu, e_ref)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("block,P", [(64, 8), (128, 8), (256, 8), (128, 2), (128, 4)])
def test_full_size_row_slice_reduce(taco, block, P):
    """The benchmark's reduce: the P row-slices of the packed [16384 x 8192]
    tensor (here the oracle's records) reduced on the GPU in one call; every
    reduced record against the oracle's reduce of the same slices (P = 8, and
    the 2- and 4-shard kernels).  Laplace
    data with outliers: the slices' decoded values cancel in many blocks, which
    tests the precision of the scales."""
    w = workloads.WORKLOADS["large_16384x8192"]
    x = w.tensor().reshape(-1)
    ref = oracle_compress_parallel(x, block)
    seg_rows = w.rows // P
    seg_bytes = taco.compressed_bytes(seg_rows, w.hidden, block)
    segs = [ref[p * seg_bytes:(p + 1) * seg_bytes] for p in range(P)]
    out = taco.reduce_shards([torch.from_numpy(s).to(DEV) for s in segs], seg_rows, w.hidden, block)
    got = out.cpu().numpy()
    assert taco.device_status() == 0
    red = oracle_reduce_parallel(segs, seg_rows * w.hidden, block)
    st = compare_records(got, red, block, u_exact=reduce_exact_u(segs, block),
                         scales_exact=exact_reduce_scales(segs, block))
    assert st["blocks"] == seg_rows * w.hidden // block
    del out
    torch.cuda.empty_cache()


def test_full_size_shard_reduce(taco):
    """Eight shards of the full [8192 x 5120] workload.  (1) Reduce in isolation:
    the GPU reduces the oracle's packed shards; every record is compared with
    the oracle's reduce of the same shards (and a sample with the oracle run
    one block at a time).  (2) The GPU decodes the oracle's reduced records,
    every element checked.  (3) The whole pipeline on the GPU (compress each
    shard, reduce, decompress) against the oracle's pipeline: relative L2 error
    of the decoded sum against the exact sum of the bf16 shards."""
    w = workloads.WORKLOADS["shard_reduce_p8_8192x5120"]
    block = 128
    xs = [w.tensor(seed=p).reshape(-1) for p in w.seeds]
    n = xs[0].size
    ref_shards = [oracle_compress_parallel(x, block) for x in xs]
    out = taco.reduce_shards([torch.from_numpy(r).to(DEV) for r in ref_shards], w.rows, w.hidden, block)
    torch.cuda.synchronize()
    assert taco.device_status() == 0
    out_np = out.cpu().numpy()
    del out
    ids = sample_blocks(n // block, 2)
    ref = oracle.reduce_shards([block_rows(r, ids, block) for r in ref_shards], ids.size * block, block)
    compare_records(block_rows(out_np, ids, block), ref, block)

    gpu_shards = [taco.compress(to_dev(x, w.rows, w.hidden), block) for x in xs]
    red = taco.reduce_shards(gpu_shards, w.rows, w.hidden, block)
    y = taco.decompress(red, w.rows, w.hidden, block)
    torch.cuda.synchronize()
    y_gpu = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    total = np.zeros(n, dtype=np.float64)
    for x in xs:
        total += (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    # The oracle's pipeline on the whole tensor, block ranges on several threads.
    from concurrent.futures import ThreadPoolExecutor
    nblk = n // block
    chunk = -(-nblk // 64)
    y_ref = np.empty(n, dtype=np.uint16)
    red_ref = np.empty(nblk * (block + 8), dtype=np.uint8)

    def run(b0):
        b1 = min(nblk, b0 + chunk)
        sl = [r[b0 * (block + 8):b1 * (block + 8)] for r in ref_shards]
        rr = oracle.reduce_shards(sl, (b1 - b0) * block, block)
        red_ref[b0 * (block + 8):b1 * (block + 8)] = rr
        y_ref[b0 * block:b1 * block] = oracle.decompress(rr, (b1 - b0) * block, block)

    with ThreadPoolExecutor(16) as ex:
        list(ex.map(run, range(0, nblk, chunk)))
    # Every reduced record of the GPU against the oracle's reduce of the same shards.
    compare_records(out_np, red_ref, block, scales_exact=exact_reduce_scales(ref_shards, block))
    # The GPU decodes the oracle's reduced records: every element.
    y_dec = bits_of(taco.decompress(torch.from_numpy(red_ref).to(DEV), w.rows, w.hidden, block))
    compare_decoded(y_dec, y_ref, block)
    yg = (y_gpu.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    yr = (y_ref.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    nt = np.linalg.norm(total)
    e_gpu = np.linalg.norm(yg - total) / nt
    e_ref = np.linalg.norm(yr - total) / nt
    assert abs(e_gpu - e_ref) <= RELL2_ATOL, (e_gpu, e_ref)


SCHEMES = [(0, 1), (0, 2), (1, 0), (2, 0), (3, 0), (2, 1)]   # (variant, code): E5M2, INT8, plain Hadamard, DS only, ASH only


@pytest.mark.parametrize("variant,code", SCHEMES)
def test_full_size_ablation_schemes(taco, variant, code):
    """The paper's ablations at the GPT-activation workload's full size
    ([8192 x 4096], block 128): every record of the GPU's compress against the
    oracle's, every element of the GPU's decode of the oracle's records, and
    the round trip's RelL2."""
    w = workloads.WORKLOADS["gpt_activation_8192x4096"]
    block = 128
    x = w.tensor().reshape(-1)
    xd = to_dev(x, w.rows, w.hidden)
    got = taco.compress(xd, block, variant=variant, code=code).cpu().numpy()
    ref = oracle_compress_parallel(x, block, variant, code)
    compare_records(got, ref, block, code=code, u_exact=exact_compress_u(x, block, variant, code),
                    scales_exact=exact_compress_scales(x, block, variant, code))
    y_ref = oracle_decompress_parallel(ref, x.size, block, variant, code)
    y_dec = bits_of(taco.decompress(torch.from_numpy(ref).to(DEV), w.rows, w.hidden, block, variant=variant,
                                    code=code))
    compare_decoded(y_dec, y_ref, block)
    y_gpu = bits_of(taco.decompress(torch.from_numpy(got).to(DEV), w.rows, w.hidden, block, variant=variant,
                                    code=code))
    assert abs(rel_l2_bf16(y_gpu, x) - rel_l2_bf16(y_ref, x)) <= RELL2_ATOL
    assert taco.device_status() == 0
    del xd
    torch.cuda.empty_cache()
