"""Seeded synthetic bf16 tensors for the five TACO workloads.

Input generation only: this package holds none of the compression method's
arithmetic.  The CUDA path (tests, benchmark, smoke check) and the CPU oracle
both take their inputs from here, and it depends on neither of them.

The values come from ``synth.c`` (built with gcc on first use): a
counter-based SplitMix64 generator keyed by (seed, stream, element index),
so any row range can be generated on its own and in parallel.  Values are
drawn in float64 and rounded to float32 and then to bf16 (nearest even each
time).  Tensors are row-major [tokens, hidden] and returned as uint16 bf16 bit
patterns.

The tensors stand in for the paper's GPT / Qwen tensor-parallel activations
and gradients, which are not available here (Section 5.1 of the TACO paper
trains on the Pile and OpenWebMath).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None
_CHUNK = 1 << 21


def build(force: bool = False) -> str:
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                            "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, f64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.synth_laplace_outliers.argtypes = [u64, i64, i64, f64, f64, f64, f64, u16p]
        lib.synth_student_t_channels.argtypes = [u64, i64, i64, i64, f64, f64, f64, u16p]
        lib.synth_gaussian_sparse.argtypes = [u64, i64, i64, f64, f64, f64, f64, u16p]
        lib.synth_small_ints.argtypes = [u64, i64, i64, i32, i32, u16p]
        lib.synth_uniform.argtypes = [u64, u64, u64]
        lib.synth_uniform.restype = f64
        for fn in (lib.synth_laplace_outliers, lib.synth_student_t_channels,
                   lib.synth_gaussian_sparse, lib.synth_small_ints):
            fn.restype = None
        _lib = lib
    return _lib


def _fill(dist: str, seed: int, hidden: int, first: int, out: np.ndarray):
    lib = _load()
    p = out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))
    n = out.size
    if dist == "laplace_outliers":
        lib.synth_laplace_outliers(seed, first, n, 1e-3, 1e-3, 0.05, 0.5, p)
    elif dist == "student_t_channels":
        lib.synth_student_t_channels(seed, first, n, hidden, 2e-3, 0.25, 8.0, p)
    elif dist == "gaussian_sparse":
        lib.synth_gaussian_sparse(seed, first, n, 1e-5, 5e-4, 1000.0, 0.2, p)
    elif dist == "small_ints":
        lib.synth_small_ints(seed, first, n, 8, -4, p)
    else:
        raise KeyError(dist)


DISTRIBUTIONS = ("laplace_outliers", "student_t_channels", "gaussian_sparse", "small_ints")


def generate(dist: str, rows: int, hidden: int, seed: int, row_start: int = 0,
             row_count: int | None = None, threads: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16, shape [row_count, hidden]) of rows
    [row_start, row_start + row_count) of the seeded [rows, hidden] tensor."""
    if dist not in DISTRIBUTIONS:
        raise KeyError(dist)
    if row_count is None:
        row_count = rows - row_start
    if row_start < 0 or row_count < 0 or row_start + row_count > rows:
        raise ValueError("row range outside the tensor")
    n = row_count * hidden
    out = np.empty(n, dtype=np.uint16)
    first = row_start * hidden
    chunks = [(c0, min(n, c0 + _CHUNK)) for c0 in range(0, n, _CHUNK)]
    if threads is None:
        threads = min(len(chunks), os.cpu_count() or 1, 16)
    if threads <= 1:
        for c0, c1 in chunks:
            _fill(dist, seed, hidden, first + c0, out[c0:c1])
    else:
        _load()
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda c: _fill(dist, seed, hidden, first + c[0], out[c[0]:c[1]]), chunks))
    return out.reshape(row_count, hidden)


def generate_rows(dist: str, hidden: int, seed: int, row_ids) -> np.ndarray:
    """bf16 bit patterns of an arbitrary set of rows, shape [len(row_ids), hidden]."""
    row_ids = np.asarray(row_ids, dtype=np.int64).reshape(-1)
    out = np.empty((row_ids.size, hidden), dtype=np.uint16)
    for i, r in enumerate(row_ids):
        _fill(dist, seed, hidden, int(r) * hidden, out[i])
    return out


def uniform(seed: int, stream: int, idx: int) -> float:
    """One uniform draw in (0, 1) of the generator (exposed for its own tests)."""
    return float(_load().synth_uniform(seed, stream, idx))


def bf16_bits_to_f32(h) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    hidden: int
    blocks: tuple
    dist: str
    seeds: tuple = (0,)
    description: str = ""

    @property
    def numel(self) -> int:
        return self.rows * self.hidden

    def tensor(self, seed: int | None = None, **kw) -> np.ndarray:
        return generate(self.dist, self.rows, self.hidden,
                        self.seeds[0] if seed is None else seed, **kw)


WORKLOADS = {
    "small_4096x1024": Workload(
        "small_4096x1024", 4096, 1024, (128,), "laplace_outliers", (0,),
        "bf16 [4096 x 1024], block 128: Laplace(0, 1e-3) bulk, 0.1% of elements "
        "replaced by +-U(0.05, 0.5) outliers; compress + decompress round trip"),
    "gpt_activation_8192x4096": Workload(
        "gpt_activation_8192x4096", 8192, 4096, (128,), "student_t_channels", (0,),
        "GPT-style TP activation, bf16 [8192 tokens (batch 4 x seq 2048) x 4096 hidden], "
        "block 128: Student-t(3) * 2e-3 * per-column log-uniform [0.25, 8) multiplier"),
    "tp_grad_8192x5120": Workload(
        "tp_grad_8192x5120", 8192, 5120, (128,), "gaussian_sparse", (0,),
        "TP backward gradient, bf16 [8192 x 5120], block 128: N(0, sd 1e-5) bulk, "
        "0.05% of entries x1000, 20% exact zeros"),
    "large_16384x8192": Workload(
        "large_16384x8192", 16384, 8192, (64, 128, 256), "laplace_outliers", (0,),
        "bf16 [16384 x 8192] (134M elements), blocks 64/128/256: Laplace(0, 1e-3) "
        "bulk + 0.1% +-U(0.05, 0.5) outliers"),
    "shard_reduce_p8_8192x5120": Workload(
        "shard_reduce_p8_8192x5120", 8192, 5120, (128,), "student_t_channels",
        tuple(range(8)),
        "P=8 shards bf16 [8192 x 5120], block 128, each the GPT-activation "
        "distribution with its own seed p = 0..7; compressed, then reduced once"),
}
