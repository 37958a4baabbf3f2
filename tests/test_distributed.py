"""The multi-rank path on CPU with the gloo backend (world size 2).

The compression operator shards without any exchange: blocks are independent,
so ranks that each compress a block-aligned slice of rows produce exactly the
records of the whole tensor (the benchmark runs one such workload per GPU,
weak scaling).  The benchmark's timing reduction takes the MAX over ranks.
The last test runs the two-shot compressed AllReduce of the TACO paper
(Section 4.4.2: compressed AlltoAll, one local reduction, compressed
AllGather) with the oracle on gloo ranks, to check that the packed record
format supports that exchange: every rank ends with the same decoded sum."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _shard_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import oracle
        import workloads
        rows, hidden, block = 64, 512, 128
        per = rows // world
        x = workloads.generate("student_t_channels", rows, hidden, seed=7, row_start=rank * per, row_count=per)
        mine = oracle.compress(x.reshape(-1), block)
        got = [None] * world
        dist.all_gather_object(got, mine)
        if rank == 0:
            full = oracle.compress(workloads.generate("student_t_channels", rows, hidden, seed=7).reshape(-1), block)
            q.put(bool(np.array_equal(np.concatenate(got), full)))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put(repr(e))


def _timing_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import bench
        vals = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        q.put((rank, vals, bench.whole_job_gbs(world, 6e9, max(vals))))
        dist.destroy_process_group()
    except Exception as e:
        q.put(repr(e))


def _two_shot_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        import oracle
        import workloads
        rows, hidden, block = 32, 256, 128
        seg = rows // world
        x = workloads.generate("laplace_outliers", rows, hidden, seed=100 + rank).reshape(rows, hidden)
        packed = oracle.compress(x.reshape(-1), block)
        seg_bytes = seg * hidden // block * (block + 8)
        # Compressed AlltoAll: segment j of every rank goes to rank j.
        outgoing = [packed[j * seg_bytes:(j + 1) * seg_bytes] for j in range(world)]
        gathered = [None] * world
        dist.all_gather_object(gathered, outgoing)
        received = [gathered[p][rank] for p in range(world)]
        # One local reduction, then a compressed AllGather of the reduced segment.
        reduced = oracle.reduce_shards(received, seg * hidden, block)
        all_reduced = [None] * world
        dist.all_gather_object(all_reduced, reduced)
        y = oracle.decompress(np.concatenate(all_reduced), rows * hidden, block)
        outs = [None] * world
        dist.all_gather_object(outs, y)
        xs = [None] * world
        dist.all_gather_object(xs, x)
        if rank == 0:
            same = all(np.array_equal(outs[0], o) for o in outs)
            exact = sum((np.asarray(v, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                        for v in xs).reshape(-1)
            got = (outs[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            rel = float(np.linalg.norm(got - exact) / np.linalg.norm(exact))
            q.put((same, rel))
        dist.destroy_process_group()
    except Exception as e:
        q.put(repr(e))


def run(worker, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = []
    try:
        for _ in range(world if worker is _timing_worker else 1):
            out.append(q.get(timeout=120))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    return out


def test_row_sharding_reproduces_whole_tensor():
    assert run(_shard_worker) == [True]


def test_timings_reduce_with_max_over_ranks():
    res = run(_timing_worker)
    assert not any(isinstance(r, str) for r in res), res
    for rank, vals, gbs in res:
        assert vals == [2.0, 5.0]
        assert abs(gbs - 2 * 6e9 / 5e-3 / 1e9) < 1e-6


def test_two_shot_allreduce_with_packed_records():
    res = run(_two_shot_worker)
    assert not isinstance(res[0], str), res
    same, rel = res[0]
    assert same
    assert rel < 0.05      # two quantisations of a bf16 sum
