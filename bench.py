#!/usr/bin/env python3
"""Benchmark of TACO's fused FP8 compression hot path on GB300.

Workload (default): bf16 [16384 x 8192] (134M elements, Laplace(0, 1e-3) bulk
with 0.1% +-U(0.05, 0.5) outliers), block 128 -- the largest single-GPU
configuration.  One step is one pass of the whole path over one tensor:

  1. taco_compress      x (bf16)            -> packed records    (Eqs. 5-10)
  2. taco_reduce_shards P = 8 row-slices of the packed tensor, taken as the P
                        compressed segments an owner receives in the two-shot
                        AllReduce, -> one reduced segment          (Section 4.4.2)
  3. taco_decompress    packed records      -> y (bf16)           (Eqs. 11-13)

Steady state.  The K steps run as CUDA graphs of C consecutive steps (C a
multiple of R with at least LAUNCHES_PER_GRAPH launches, and one graph for the
K mod C steps left), replayed back to back: each replay boundary leaves the GPU
idle for a few microseconds, which a graph of C steps pays once.  Inputs rotate
over R buffer sets (R x the bytes of one set >= 3 x L2) and the three kernels
of step k work on different sets: compress on set k, the reduce on the packed
records of set k-2 and decompress on those of set k-3 (k mod R), so every
kernel reads data last written at least two kernels and some hundreds of MB of
traffic earlier, from HBM, and the deferred write-back of every kernel's output
is paid inside the timed region.  Each kernel's own average launch duration is
timed the same way: graphs of at least LAUNCHES_PER_GRAPH back-to-back launches
of that kernel alone over the rotating sets, replayed.

Metric (`value`): compress/decompress GB/s of bf16 input = 2 x 2N bytes (the
bf16 tensor compressed plus the bf16 tensor decompressed) over the sum of the
two kernels' average launch durations.  The whole step (with the reduce) is
reported under `step`; the same workload at the other block sizes under
`blocks`; the reduce of 8 full-size [8192 x 5120] shards under
`reduce_full_shards`; the reduce of the tensor split into 2, 4 and 16 shards
under `reduce_shard_counts`.  The roofline object reports the dominant kernel's
algorithmic bytes per launch over its average duration against the measured
HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl taco|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
seed (weak scaling, no collective on the data path); timings are reduced with
MAX over ranks and rank 0 prints the JSON line.  `--impl reference` times the
CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "compress/decompress GB/s of bf16 input; % of GB300 HBM roofline"
UNIT = "GB/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "compress": "fp8_compression_tensor_gb300/csrc/taco_compress.cu",
    "decompress": "fp8_compression_tensor_gb300/csrc/taco_decompress.cu",
    "reduce": "fp8_compression_tensor_gb300/csrc/taco_reduce.cu",
}
FALLBACK_HBM_GBS = 6800.0
# Launches per captured graph (at least): a replay boundary idles the GPU for
# about 4 us, which would otherwise be charged to the launches of one replay.
LAUNCHES_PER_GRAPH = 32


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["taco", "reference"], default="taco")
    ap.add_argument("--workload", default="large_16384x8192", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--block", type=int, default=128)
    ap.add_argument("--shards", type=int, default=8)
    ap.add_argument("--variant", default="ash_ds", choices=["ash_ds", "hadamard_ds", "ds_only", "ash_only"],
                    help="ablation variant (the method is ash_ds)")
    ap.add_argument("--code", default="e4m3", choices=["e4m3", "e5m2", "int8"],
                    help="code format (the method is e4m3)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other block sizes and the full-size shard reduce (extra keys)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------

def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and blank space, so that editing a
    comment does not invalidate DRAM counters taken on the same code."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c == '"':                        # string literal (PTX text): kept verbatim
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(rel: str) -> str:
    """Hash of a kernel's code (its .cu file and the shared headers), comments excluded."""
    h = hashlib.sha256()
    for p in (rel, "fp8_compression_tensor_gb300/csrc/taco_device.cuh",
              "fp8_compression_tensor_gb300/csrc/taco_tcgen05.cuh",
              "fp8_compression_tensor_gb300/csrc/taco_sched.cuh",
              "fp8_compression_tensor_gb300/csrc/taco_kernels.h"):
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def traffic_for(op: str, workload: str, block: int):
    """DRAM bytes per launch from a committed ncu capture (dict with the bytes
    read and written and how they were taken), if the kernel's source has not
    changed since the capture; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t[op][f"{workload}/b{block}"]
        if e["source_hash"] != source_hash(KERNEL_SOURCES[op]):
            return None
        return e
    except Exception:
        return None


class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid):
        self.uuid = device_uuid
        self.samples = []
        self.proc = None
        self.thread = None
        self.error = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # nvidia-smi missing
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": self.error}
        rows = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not rows:
            rows = [p for (_, p) in self.samples]
            window = "whole run"
        else:
            window = "timed region"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        busy = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in busy if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window": window,
                "power_w_max": max((num(r[3]) or 0) for r in rows) if rows else None}


# ---------------------------------------------------------------------------
# Oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def oracle_op_times(x_bits: np.ndarray, block: int, shards: int, threads: int) -> dict:
    """The oracle's compress, reduce of the P row-slices and decompress over
    x_bits, each split into block ranges across `threads`: their wall times
    (seconds) and outputs (packed records, reduced segment, decoded bf16)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    x = np.ascontiguousarray(x_bits).reshape(-1)
    n = x.size
    nblk = n // block
    rec = block + 8
    seg_blk = nblk // shards
    packed = np.empty(nblk * rec, dtype=np.uint8)
    y = np.empty(n, dtype=np.uint16)
    red = np.empty(seg_blk * rec, dtype=np.uint8)

    def ranges(total):
        c = max(1, -(-total // (4 * threads)))
        return [(b, min(total, b + c)) for b in range(0, total, c)]

    def comp(r):
        b0, b1 = r
        packed[b0 * rec:b1 * rec] = oracle.compress(x[b0 * block:b1 * block], block)

    def reduce_(r):
        b0, b1 = r
        segs = [packed[(p * seg_blk + b0) * rec:(p * seg_blk + b1) * rec] for p in range(shards)]
        red[b0 * rec:b1 * rec] = oracle.reduce_shards(segs, (b1 - b0) * block, block)

    def decomp(r):
        b0, b1 = r
        y[b0 * block:b1 * block] = oracle.decompress(packed[b0 * rec:b1 * rec], (b1 - b0) * block, block)

    t = {}
    with ThreadPoolExecutor(threads) as ex:
        for name, fn, total in (("compress", comp, nblk), ("reduce", reduce_, seg_blk),
                                ("decompress", decomp, nblk)):
            t0 = time.perf_counter()
            list(ex.map(fn, ranges(total)))
            t[name] = time.perf_counter() - t0
    return {"seconds": t, "packed": packed, "reduced": red, "y": y}


def oracle_metric(n: int, t: dict) -> float:
    """The metric for one oracle pass over n elements: GB/s of bf16 input of
    compress and decompress (2 x 2n bytes over their summed time)."""
    return 4.0 * n / (t["compress"] + t["decompress"]) / 1e9


def oracle_build_info() -> str:
    """Compiler and flags the oracle library is built with."""
    import oracle
    return "gcc " + " ".join(f for f in oracle.CFLAGS if f not in ("-fPIC", "-shared"))


def max_over_ranks(values, device=None):
    """Element-wise MAX of a list of floats over all ranks (identity on one
    process); timings are reduced this way so that the slowest rank sets the
    whole job's time."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_gbs(world: int, bytes_per_rank_step: float, ms_per_step: float) -> float:
    """Aggregate GB/s over all ranks: every rank processes its own workload
    (weak scaling) in at most the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def sample_rows_for(w, block, shards, threads, budget_s):
    """Rows of the workload whose oracle pass (compress, reduce, decompress)
    takes about budget_s seconds (a multiple of `shards` rows, at least
    `shards`)."""
    probe_rows = max(shards, min(w.rows, 64 * shards))
    x = w.tensor(row_count=probe_rows)
    t = sum(oracle_op_times(x, block, shards, threads)["seconds"].values())
    rows = int(probe_rows * budget_s / max(t, 1e-6))
    rows = max(shards, min(w.rows, rows)) // shards * shards
    return rows


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores, on a row sample of
    the same workload; each step is one oracle pass (compress, reduce of the
    P row-slices, decompress), and `value` is the same metric as the GPU
    arm's (compress/decompress GB/s of bf16 input)."""
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    block, shards = args.block, args.shards
    threads = host_threads()
    # Size each step so that warm-up plus timed steps stay within ~2 minutes.
    per_step_budget = min(15.0, 120.0 / max(1, args.steps + args.warmup))
    rows = sample_rows_for(w, block, shards, threads, per_step_budget)
    x = w.tensor(row_count=rows)
    for _ in range(args.warmup):
        oracle_op_times(x, block, shards, threads)
    runs = [oracle_op_times(x, block, shards, threads)["seconds"] for _ in range(args.steps)]
    n = x.size
    t = {k: sum(r[k] for r in runs) / len(runs) for k in runs[0]}
    value = oracle_metric(n, t)
    step_s = sum(t.values())
    sample = (f"rows [0, {rows}) of the {w.rows}x{w.hidden} tensor ({n} elements) per step: "
              f"compress, reduce of {shards} row-slices, decompress; block ranges split over {threads} threads; "
              f"value = 2 x 2n bytes over the mean compress + decompress time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "hidden": w.hidden, "block": block,
                   "reduce_shards": shards, "sample_rows": rows},
        "ops_ms": {k: v * 1e3 for k, v in t.items()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model(), "compiler": oracle_build_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_taco(args, rank, world):
    import torch
    import torch.distributed as dist
    import fp8_compression_tensor_gb300 as taco

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    block, P = args.block, args.shards
    rows, hidden = w.rows, w.hidden
    if rows % P:
        raise SystemExit(f"rows {rows} not divisible by {P} shards")
    n = rows * hidden
    seg_rows = rows // P
    rec = block + 8
    nbytes = taco.compressed_bytes(rows, hidden, block)
    seg_bytes = taco.compressed_bytes(seg_rows, hidden, block)

    x_host_bits = w.tensor(seed=w.seeds[0] + rank).reshape(rows, hidden)
    x_pinned = torch.from_numpy(x_host_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20)) or (128 << 20)
    set_bytes = 2 * n + nbytes + seg_bytes + 2 * n
    R = max(4, -(-3 * l2 // set_bytes))
    xs = [x_pinned.to(dev) for _ in range(R)]
    packs = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(R)]
    reds = [torch.empty(seg_bytes, dtype=torch.uint8, device=dev) for _ in range(R)]
    ys = [torch.empty((rows, hidden), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    segs = [[packs[r][p * seg_bytes:(p + 1) * seg_bytes] for p in range(P)] for r in range(R)]
    stream = torch.cuda.Stream(dev)

    scheme = {"variant": args.variant, "code": args.code}

    def op_compress(r, st=None):
        taco.compress(xs[r], block, out=packs[r], stream=st or stream, **scheme)

    def op_reduce(r, st=None):
        taco.reduce_shards(segs[r], seg_rows, hidden, block, out=reds[r], stream=st or stream, **scheme)

    def op_decompress(r, st=None):
        taco.decompress(packs[r], rows, hidden, block, out=ys[r], stream=st or stream, **scheme)

    # A cycle of steps as a graph with one branch per kernel kind and an
    # edge only where data flows (compress -> reduce / decompress of the same
    # set, and a set's next compress after the reads of its records): the
    # three kernels of a step work on different buffer sets (micro-batches),
    # so one kernel's tail overlaps the next kernel's start.
    branch = {"C": torch.cuda.Stream(dev), "R": torch.cuda.Stream(dev), "D": torch.cuda.Stream(dev)}

    def cycle_with_data_edges(steps):
        ops = []
        for k in range(steps):
            ops += [("C", k % R), ("R", (k - 2) % R), ("D", (k - 3) % R)]
        for st in branch.values():
            st.wait_stream(stream)
        last_write, readers = {}, {}
        for kind, r in ops:
            st = branch[kind]
            reads = [("x", r)] if kind == "C" else [("packed", r)]
            writes = [("packed", r)] if kind == "C" else [("reduced", r)] if kind == "R" else [("y", r)]
            for buf in reads + writes:
                if buf in last_write:
                    st.wait_event(last_write[buf])
            for buf in writes:
                for e in readers.get(buf, []):
                    st.wait_event(e)
            {"C": op_compress, "R": op_reduce, "D": op_decompress}[kind](r, st)
            done = torch.cuda.Event()
            done.record(st)
            for buf in reads:
                readers.setdefault(buf, []).append(done)
            for buf in writes:
                last_write[buf] = done
                readers[buf] = []
        for st in branch.values():
            stream.wait_stream(st)

    def step(k):
        op_compress(k % R)
        op_reduce((k - 2) % R)
        op_decompress((k - 3) % R)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    # Graphs of L = M x R launches (M passes over the rotating sets).
    K = args.steps
    M, L, C = graph_plan(K, R)

    def capture_solo(fn):
        return capture(lambda: [fn(r) for _ in range(M) for r in range(R)])

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for r in range(R):          # every set holds valid records before the skewed steps read them
            op_compress(r)
        for k in range(R):
            step(k)
        stream.synchronize()
        step_graphs = [capture(lambda k=k: step(k)) for k in range(R)]
        cycle_graph = capture(lambda: cycle_with_data_edges(C))   # C steps, the R sets C / R times each
        tail_graph = capture(lambda: cycle_with_data_edges(K % C)) if K % C else None
        solo_graphs = {name: capture_solo(fn)
                       for name, fn in (("compress", op_compress), ("reduce", op_reduce),
                                        ("decompress", op_decompress))}

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    if not args.no_clocks:
        sampler.start()

    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            step_graphs[k % R].replay()
    barrier()
    taco.device_status(stream=stream)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(K // C):
            cycle_graph.replay()
        if tail_graph is not None:
            tail_graph.replay()
        ev1.record(stream)
    barrier()
    t_wall1 = time.time()
    flags = taco.device_status(stream=stream)
    ms_step = max_over_ranks([ev0.elapsed_time(ev1) / K], device=dev)[0]

    names = ("compress", "reduce", "decompress")
    solo = time_solo(solo_graphs, stream, L, K, dev)
    solo_ms = {k: solo[k]["ms"] for k in names}
    t_wall2 = time.time()            # the clock record covers the steps and the per-kernel timings

    peak, peak_src = measured_peak()
    alg = {"compress": 2 * n + nbytes, "reduce": P * seg_bytes + seg_bytes, "decompress": nbytes + 2 * n}

    def op_line(op, t, alg_bytes, n_el):
        sec = t["ms"] * 1e-3
        return {"ms": t["ms"], "bf16_gbs": 2 * n_el / sec / 1e9, "hbm_gbs": alg_bytes / sec / 1e9,
                "frac_of_measured_hbm": alg_bytes / sec / 1e9 / peak,
                "frac_of_nominal_8tbs": alg_bytes / sec / 1e9 / 8000.0, "algorithmic_bytes": alg_bytes,
                "launches_timed": t["launches"], "ms_median_of_groups": t["median"], "ms_min_of_groups": t["min"],
                "groups": t["groups"]}

    ops = {op: op_line(op, solo[op], alg[op], n) for op in names}
    # The reduce's logical bf16 input is P segments of N / P elements: N.
    value = whole_job_gbs(world, 4.0 * n, solo_ms["compress"] + solo_ms["decompress"])

    # Extra keys: the same workload at its other block sizes, and the reduce
    # of 8 full-size shards (the owner's local step on the P-seed workload).
    blocks = None
    full_reduce = None
    shard_counts = None
    if not args.no_extras:
        blocks = {}
        for b in w.blocks:
            if b == block:
                continue
            nb = taco.compressed_bytes(rows, hidden, b)
            sb = taco.compressed_bytes(seg_rows, hidden, b)
            pk_b = [torch.empty(nb, dtype=torch.uint8, device=dev) for _ in range(R)]
            rd_b = [torch.empty(sb, dtype=torch.uint8, device=dev) for _ in range(R)]
            sg_b = [[pk_b[r][p * sb:(p + 1) * sb] for p in range(P)] for r in range(R)]
            fns = {"compress": lambda r, b=b, pk_b=pk_b: taco.compress(xs[r], b, out=pk_b[r], stream=stream,
                                                                        **scheme),
                   "reduce": lambda r, b=b, sg_b=sg_b, rd_b=rd_b: taco.reduce_shards(
                       sg_b[r], seg_rows, hidden, b, out=rd_b[r], stream=stream, **scheme),
                   "decompress": lambda r, b=b, pk_b=pk_b: taco.decompress(pk_b[r], rows, hidden, b, out=ys[r],
                                                                          stream=stream, **scheme)}
            with torch.cuda.stream(stream):
                for r in range(R):
                    fns["compress"](r)
                graphs = {name: capture_solo(fns[name]) for name in names}
            tb = time_solo(graphs, stream, L, K, dev)
            alg_b = {"compress": 2 * n + nb, "reduce": (P + 1) * sb, "decompress": nb + 2 * n}
            entry = {op: op_line(op, tb[op], alg_b[op], n) for op in names}
            entry["value"] = whole_job_gbs(world, 4.0 * n, tb["compress"]["ms"] + tb["decompress"]["ms"])
            blocks[str(b)] = entry
            del pk_b, rd_b, sg_b, graphs
            torch.cuda.empty_cache()
        full_reduce = time_full_shard_reduce(taco, workloads.WORKLOADS["shard_reduce_p8_8192x5120"], block, scheme,
                                             stream, dev, capture, peak)
        # The reduce of the same packed tensor split into other shard counts
        # (an owner's step at tensor-parallel degree 2, 4 and 16).
        shard_counts = {}
        for P2 in (2, 4, 16):
            if P2 == P or rows % P2:
                continue
            sr2 = rows // P2
            sb2 = taco.compressed_bytes(sr2, hidden, block)
            outs2 = [torch.empty(sb2, dtype=torch.uint8, device=dev) for _ in range(R)]
            segs2 = [[packs[r][p * sb2:(p + 1) * sb2] for p in range(P2)] for r in range(R)]
            with torch.cuda.stream(stream):
                for r in range(R):
                    op_compress(r)
                g2 = {"reduce": capture_solo(lambda r: taco.reduce_shards(segs2[r], sr2, hidden, block,
                                                                          out=outs2[r], stream=stream, **scheme))}
            t2 = time_solo(g2, stream, L, K, dev)["reduce"]
            shard_counts[str(P2)] = op_line("reduce", t2, (P2 + 1) * sb2, n)
            del outs2, segs2, g2
        torch.cuda.empty_cache()
    x, packed, reduced, y = xs[0], packs[0], reds[0], ys[0]

    # Reconstruction error of the round trip (paper Eq. 21), fp64 over the tensor.
    with torch.cuda.stream(stream):
        op_compress(0)
        op_decompress(0)
    stream.synchronize()
    xd, yd = x.double(), y.double()
    rel_l2 = float(torch.linalg.vector_norm(yd - xd) / torch.linalg.vector_norm(xd))
    del xd, yd

    # End to end through the public API with host buffers: pinned H2D of the
    # step's input, the three calls, D2H of the decompressed tensor and of
    # the reduced segment, every step.
    e2e = None
    if not args.no_e2e:
        # Through the public API with host buffers, every step: the input from
        # pinned host memory, the three calls, the decompressed tensor and the
        # reduced segment back to pinned host memory.  Copies in and out run on
        # their own streams over two device buffer sets, so step k's upload,
        # step k-1's kernels and step k-2's download overlap (steady state).
        y_pinned = [torch.empty((rows, hidden), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        r_pinned = [torch.empty(seg_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("up", "done", "down")}

        def e2e_step(k):
            b = k % 2
            xd, pk, rd, yd = xs[b], packs[b], reds[b], ys[b]
            sg = segs[b]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev["done"][b])             # step k-2's kernels have read xs[b]
                xd.view(-1).copy_(x_pinned.view(-1), non_blocking=True)
                ev["up"][b].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev["up"][b])
                if k >= 2:
                    stream.wait_event(ev["down"][b])           # step k-2's results have left ys[b], reds[b]
                taco.compress(xd, block, out=pk, stream=stream, **scheme)
                taco.reduce_shards(sg, seg_rows, hidden, block, out=rd, stream=stream, **scheme)
                taco.decompress(pk, rows, hidden, block, out=yd, stream=stream, **scheme)
                ev["done"][b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["done"][b])
                y_pinned[b].copy_(yd, non_blocking=True)
                r_pinned[b].copy_(rd, non_blocking=True)
                ev["down"][b].record(s_out)

        for k in range(max(2, min(args.warmup, 6))):
            e2e_step(k)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k_e2e = max(1, min(K, 100))
        e0.record(s_in)
        for k in range(k_e2e):
            e2e_step(k)
        e1.record(s_out)
        barrier()
        ms = max_over_ranks([e0.elapsed_time(e1) / k_e2e], device=dev)[0]
        e2e = {"value": whole_job_gbs(world, 4.0 * n, ms), "unit": UNIT, "ms_per_step": ms,
               "steps": k_e2e, "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 2 * n + seg_bytes,
               "what": "compress + reduce + decompress through the public API with the input uploaded from and "
                       "the decompressed tensor and reduced segment downloaded to pinned host memory every step; "
                       "value = 2 x 2N bf16 bytes per step over the step time",
               "overlap": "uploads, kernels and downloads on three streams, two buffer sets"}

    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall2) if not args.no_clocks else None
    flags |= taco.device_status(stream=stream)

    cpu = None
    parity = None
    if not args.no_cpu_baseline:
        threads = host_threads()
        # About 20 s of CPU work (threads x wall seconds): a row sample of the
        # workload, its oracle pass repeated while the whole tensor is too
        # small to fill the budget.
        budget = max(1.0, 20.0 / threads)
        srows = sample_rows_for(w, block, P, threads, budget)
        xsmp = x_host_bits[:srows]
        runs = [oracle_op_times(xsmp, block, P, threads)]
        while sum(sum(r["seconds"].values()) for r in runs) < budget:
            runs.append(oracle_op_times(xsmp, block, P, threads))
        t_cpu = {k: sum(r["seconds"][k] for r in runs) / len(runs) for k in runs[0]["seconds"]}
        # The same oracle on one core, on a sample of about 2 s.
        rows1 = sample_rows_for(w, block, P, 1, 2.0)
        t1 = oracle_op_times(x_host_bits[:rows1], block, P, 1)["seconds"]
        cpu = {"value": oracle_metric(xsmp.size, t_cpu), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"rows [0, {srows}) of the {rows}x{hidden} tensor: {len(runs)} oracle pass(es) "
                         f"(compress, reduce of {P} row-slices, decompress), block ranges split over "
                         f"{threads} threads; value = 2 x 2n bytes over the mean compress + decompress time",
               "seconds": sum(sum(r["seconds"].values()) for r in runs),
               "ops_ms": {k: v * 1e3 for k, v in t_cpu.items()},
               "single_core": {"value": oracle_metric(rows1 * hidden, t1), "unit": UNIT, "cores": 1,
                               "sample": f"rows [0, {rows1}): one oracle pass on one thread"},
               "cpu_model": cpu_model(), "compiler": oracle_build_info()}
        # Parity of the timed kernels against the oracle's outputs on the same
        # sample rows (outside every timed region).
        parity = parity_against_oracle(taco, runs[-1], xsmp, block, P, scheme, stream, dev)

    if rank != 0:
        return

    dom = max(("compress", "decompress", "reduce"), key=lambda k: solo_ms[k])
    achieved = alg[dom] / (solo_ms[dom] * 1e-3) / 1e9
    tr = traffic_for(dom, w.name, block)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": peak_src,
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "traffic_read": tr["dram_read_per_launch"] if tr else None,
                "traffic_write": tr["dram_write_per_launch"] if tr else None,
                "traffic_how": tr["how"] if tr else "no capture of the current kernel code",
                "algorithmic_bytes_per_launch": alg[dom],
                "duration": (f"mean of {solo[dom]['launches']} back-to-back launches of the kernel alone (graphs "
                             f"of {L} launches over the {R} rotating sets, replayed), CUDA events on its stream")}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "rows": rows, "hidden": hidden, "block": block, "reduce_shards": P,
                   "variant": args.variant, "code": args.code,
                   "value": "2 x 2N bytes of bf16 input (compressed and decompressed) over the summed mean "
                            "launch times of compress and decompress, each timed alone back to back",
                   "step": "compress + reduce_shards(P row-slices of the packed tensor) + decompress",
                   "l2": (f"no flush; inputs larger than L2: {R} rotating buffer sets of {set_bytes / 1e6:.1f} MB "
                          f"(L2 {l2 / 1e6:.0f} MB); step k compresses set k, reduces set k-2, decompresses "
                          f"set k-3; graph replays (one graph per {C} steps and one for the K mod {C} left, a "
                          f"branch per kernel kind with edges only for data dependencies, so kernels of "
                          f"different sets overlap at their boundaries), one CUDA-event pair around the K steps"),
                   "buffer_sets": R, "steps_per_graph": C, "launches_per_graph": L,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "step": {"ms": ms_step, "gbs_6n": whole_job_gbs(world, 6.0 * n, ms_step),
                 "what": "the K timed steps: 6N bytes per step (2N compressed + 2N logical bf16 of the reduced "
                         "segments + 2N decompressed) over the step time"},
        "ops": ops,
        "ops_sum_ms": sum(solo_ms.values()),
        "blocks": blocks,
        "reduce_full_shards": full_reduce,
        "reduce_shard_counts": shard_counts,
        "quality": {"rel_l2_round_trip": rel_l2},
        "parity": parity,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "device_fault_flags": flags,
        "wall_s_timed": t_wall1 - t_wall0,
        "gpu": props.name,
    }
    print(json.dumps(line), flush=True)


def graph_plan(K: int, R: int, min_launches: int = LAUNCHES_PER_GRAPH):
    """How the timed work is cut into graphs, over R rotating buffer sets:
    M passes over the sets per per-kernel graph (L = M x R >= min_launches
    launches), and C steps per step graph (a multiple of R, at most L); the K
    steps run as K // C replays of the C-step graph and one graph of the
    K mod C steps left."""
    if K < 1 or R < 1:
        raise ValueError("need K >= 1 steps and R >= 1 buffer sets")
    M = -(-min_launches // R)
    L = M * R
    C = min(L, max(R, K // R * R))
    return M, L, C


def time_solo(graphs: dict, stream, L: int, K: int, dev) -> dict:
    """Each kernel alone: its graph of L back-to-back launches over the
    rotating sets, replayed (about min(1000, 2K) launches in all); events
    split the replays into G groups.  Per kernel: the mean over all launches
    (ms), the median and minimum of the groups' per-launch means, MAX over
    ranks."""
    import torch
    reps = max(4, min(1000, 2 * K) // L)
    G = min(10, reps)
    reps = reps // G * G
    out = {}
    with torch.cuda.stream(stream):
        for name, g in graphs.items():
            for _ in range(2):
                g.replay()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(G + 1)]
            evs[0].record(stream)
            for j in range(G):
                for _ in range(reps // G):
                    g.replay()
                evs[j + 1].record(stream)
            stream.synchronize()
            per = [evs[j].elapsed_time(evs[j + 1]) / (reps // G * L) for j in range(G)]
            t = max_over_ranks([evs[0].elapsed_time(evs[G]) / (reps * L), statistics.median(per), min(per)],
                               device=dev)
            out[name] = {"ms": t[0], "median": t[1], "min": t[2], "launches": reps * L, "groups": G,
                         "launches_per_graph": L}
    return out


def time_full_shard_reduce(taco, wf, block, scheme, stream, dev, capture, peak):
    """The reduce of P full-size packed shards (the P-seed workload: each shard
    its own seeded tensor, compressed on the GPU): a graph of
    LAUNCHES_PER_GRAPH back-to-back launches on the same shards (401 MB of
    traffic a launch, three times L2), replayed."""
    import torch
    Pf = len(wf.seeds)
    rows, hidden = wf.rows, wf.hidden
    n = rows * hidden
    nbytes = taco.compressed_bytes(rows, hidden, block)
    full = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(Pf)]
    full_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for p_, sd in enumerate(wf.seeds):
            xf = torch.from_numpy(wf.tensor(seed=sd).view(np.int16)).view(torch.bfloat16).to(dev).view(rows, hidden)
            taco.compress(xf, block, out=full[p_], stream=stream, **scheme)
            stream.synchronize()
            del xf
        Lf = LAUNCHES_PER_GRAPH
        g_full = capture(lambda: [taco.reduce_shards(full, rows, hidden, block, out=full_out, stream=stream,
                                                     **scheme) for _ in range(Lf)])
        g_full.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps_f = 8
        a.record(stream)
        for _ in range(reps_f):
            g_full.replay()
        b.record(stream)
        stream.synchronize()
    ms_f = max_over_ranks([a.elapsed_time(b) / (reps_f * Lf)], device=dev)[0]
    alg_f = (Pf + 1) * nbytes
    return {"workload": wf.name, "ms": ms_f, "shards": Pf, "block": block, "algorithmic_bytes": alg_f,
            "hbm_gbs": alg_f / ms_f / 1e6, "frac_of_measured_hbm": alg_f / ms_f / 1e6 / peak,
            "frac_of_nominal_8tbs": alg_f / ms_f / 1e6 / 8000.0, "logical_bf16_gbs": Pf * 2 * n / ms_f / 1e6,
            "launches": reps_f * Lf, "launches_per_graph": Lf,
            "what": f"reduce of {Pf} full-size packed [{rows} x {hidden}] shards (seeds {list(wf.seeds)}), "
                    f"graphs of {Lf} back-to-back launches on the same input, replayed"}


def parity_against_oracle(taco, run, x_bits, block, P, scheme, stream, dev) -> dict:
    """Parity statistics of the GPU kernels against the oracle's outputs of
    one timed oracle pass (`run`, from oracle_op_times) on the same sample
    rows: the GPU's records against the oracle's, the GPU's decode of the
    oracle's records, and the GPU's reduce of the oracle's P row-slices (the
    stats of tests/parity.py, reported, not asserted)."""
    import torch
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import bf16_to_f64, exact_compress_quantities
    from parity import compare_decoded, compare_records, exact_compress_scales, exact_reduce_scales, reduce_exact_u
    if scheme["variant"] != "ash_ds" or scheme["code"] != "e4m3":
        return None
    rows, hidden = x_bits.shape
    nblk = x_bits.size // block
    rec = block + 8
    seg_rows = rows // P
    seg_bytes = seg_rows * hidden // block * rec
    with torch.cuda.stream(stream):
        xd = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).to(dev)
        got = taco.compress(xd, block, stream=stream).cpu().numpy()
        ref_dev = torch.from_numpy(run["packed"]).to(dev)
        y = taco.decompress(ref_dev, rows, hidden, block, stream=stream)
        segs = [ref_dev[p * seg_bytes:(p + 1) * seg_bytes] for p in range(P)]
        red = taco.reduce_shards(segs, seg_rows, hidden, block, stream=stream).cpu().numpy()
        y_np = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    _, _, u, _ = exact_compress_quantities(bf16_to_f64(x_bits.reshape(-1)), block)
    c = compare_records(got, run["packed"], block, check=False, u_exact=u,
                        scales_exact=exact_compress_scales(x_bits.reshape(-1), block))
    segs_np = [run["packed"][p * seg_bytes:(p + 1) * seg_bytes] for p in range(P)]
    r = compare_records(red, run["reduced"], block, check=False, u_exact=reduce_exact_u(segs_np, block),
                        scales_exact=exact_reduce_scales(segs_np, block))
    d = compare_decoded(y_np, run["y"], block, check=False)
    keep = ("code_mismatch_frac", "code_mismatches", "mismatch_budget", "tie_mismatches", "code_max_step",
            "alpha_max_rel", "s_max_rel", "alpha_max_rel_vs_ref", "s_max_rel_vs_ref", "scales_closer_to_exact",
            "s_zero_mismatch")
    return {"sample_blocks": nblk,
            "compress": {k: c[k] for k in keep},
            "reduce": {k: r[k] for k in keep},
            "decompress": {"bf16_mismatch_frac": d["mismatch_frac"], "beyond_one_step": d["bad"]},
            "bar": "scales 1e-6 relative (or within 1e-6 of the real-arithmetic value and closer to it than the "
                   "oracle's); codes identical except <= 1e-4 of elements (+ twice the rounding ties the oracle "
                   "itself rounds away from the exact value), one step apart; decoded bf16 within one step where "
                   "FP32 noise of the block scale reaches a midpoint"}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_taco(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
