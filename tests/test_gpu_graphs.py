"""Stream-ordering and CUDA-graph behaviour of the C ABI on the GPU.

Every kernel starts (programmatic dependent launch) while the previous kernel
in the stream drains, prefetches its first tiles into L2 and only then waits
for that kernel; it must still read the data the previous kernel wrote.  The
kernels are deterministic, so every check here is bit-exact:

* a chain in which each call reads the output of the call just before it, on
  one stream with no synchronisation, equals the same chain with a device
  synchronisation between the calls;
* compress -> shard reduce -> decompress captured in a CUDA graph and replayed
  on new input contents (the graph's kernels read the buffers, not captured
  values) equals the eager calls on the same input;
* chains on three streams running at the same time equal each chain run
  alone.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def bf16_input(dist, rows, hidden, seed):
    x = workloads.generate(dist, rows, hidden, seed=seed)
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).reshape(rows, hidden).to(DEV)


def chain(taco, x, block, stream, sync):
    """x -> compress -> decompress -> compress -> decompress -> compress."""
    outs = []
    cur = x
    for k in range(5):
        if k % 2 == 0:
            cur = taco.compress(cur, block, stream=stream)
        else:
            cur = taco.decompress(cur, x.shape[0], x.shape[1], block, stream=stream)
        outs.append(cur)
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return [o.view(torch.uint8).cpu().numpy() if o.dtype == torch.uint8 else o.view(torch.int16).cpu().numpy()
            for o in outs]


@pytest.mark.parametrize("block", [64, 128, 256, 512])
def test_back_to_back_dependent_calls(taco, block):
    rows, hidden = 4096, 2048          # 4096 tiles at B = 64: many CTAs per SM
    x = bf16_input("student_t_channels", rows, hidden, seed=11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fast = chain(taco, x, block, s, sync=False)
    ref = chain(taco, x, block, s, sync=True)
    for k, (a, b) in enumerate(zip(fast, ref)):
        assert np.array_equal(a, b), f"call {k} of the chain differs without synchronisation"
    assert taco.device_status() == 0


def test_graph_replay_matches_eager(taco):
    rows, hidden, block, P = 8192, 1024, 128, 8
    seg_rows = rows // P
    seg = taco.compressed_bytes(seg_rows, hidden, block)
    x = torch.empty(rows, hidden, dtype=torch.bfloat16, device=DEV)
    packed = torch.empty(taco.compressed_bytes(rows, hidden, block), dtype=torch.uint8, device=DEV)
    red = torch.empty(seg, dtype=torch.uint8, device=DEV)
    y = torch.empty(rows, hidden, dtype=torch.bfloat16, device=DEV)
    segs = [packed[p * seg:(p + 1) * seg] for p in range(P)]

    def step(stream):
        taco.compress(x, block, out=packed, stream=stream)
        taco.reduce_shards(segs, seg_rows, hidden, block, out=red, stream=stream)
        taco.decompress(packed, rows, hidden, block, out=y, stream=stream)

    def snapshot():
        torch.cuda.synchronize()
        return packed.cpu().numpy().copy(), red.cpu().numpy().copy(), y.view(torch.int16).cpu().numpy().copy()

    s = torch.cuda.Stream()
    x.copy_(bf16_input("laplace_outliers", rows, hidden, seed=3))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step(s)                        # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    torch.cuda.synchronize()

    for seed, dist in ((5, "student_t_channels"), (6, "gaussian_sparse"), (5, "student_t_channels")):
        x.copy_(bf16_input(dist, rows, hidden, seed=seed))
        packed.zero_()
        red.zero_()
        y.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            step(s)
        eager = snapshot()
        packed.fill_(0xAB)
        red.fill_(0xAB)
        y.zero_()
        torch.cuda.synchronize()
        g.replay()
        graphed = snapshot()
        for name, a, b in zip(("packed", "reduced", "decompressed"), graphed, eager):
            assert np.array_equal(a, b), f"graph replay differs from the eager calls in {name} ({dist}, seed {seed})"
    assert taco.device_status() == 0


def test_concurrent_streams_match_sequential(taco):
    """Calls on different streams may run at the same time on the GPU (each
    grid schedules its own tiles); every output equals the one computed alone."""
    rows, hidden, P = 4096, 2048, 4
    seg_rows = rows // P
    seg = taco.compressed_bytes(seg_rows, hidden, 128)
    xs = [bf16_input(d, rows, hidden, seed=20 + i)
          for i, d in enumerate(("student_t_channels", "laplace_outliers", "gaussian_sparse"))]
    blocks = (128, 64, 256)

    def chain(x, block, stream):
        p = taco.compress(x, block, stream=stream)
        y = taco.decompress(p, rows, hidden, block, stream=stream)
        r = None
        if block == 128:
            r = taco.reduce_shards([p[i * seg:(i + 1) * seg] for i in range(P)], seg_rows, hidden, block,
                                   stream=stream)
        return p, y, r

    def host(outs):
        return [None if t is None else (t.cpu().numpy() if t.dtype == torch.uint8
                                        else t.view(torch.int16).cpu().numpy()) for t in outs]

    ref = []
    for x, b in zip(xs, blocks):
        ref.append(host(chain(x, b, torch.cuda.current_stream())))
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in xs]
    torch.cuda.synchronize()
    for _ in range(3):
        outs = []
        for x, b, s in zip(xs, blocks, streams):
            with torch.cuda.stream(s):
                outs.append(chain(x, b, s))
        torch.cuda.synchronize()
        for k, (o, r) in enumerate(zip(outs, ref)):
            for name, a, b in zip(("packed", "decompressed", "reduced"), host(o), r):
                assert (a is None) == (b is None)
                if a is not None:
                    assert np.array_equal(a, b), f"stream {k}: {name} differs from the call made alone"
    assert taco.device_status() == 0
