"""CPU oracle for TACO's fused FP8 compression operator (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  The CUDA library and
its Python binding never import, link or call it, and it shares no code with
them.  The arithmetic lives in ``taco_oracle.c`` (plain single-threaded C,
built with ``-O2 -ffp-contract=off``); this module builds it with gcc on first
use and wraps it with ctypes and numpy.

Every function follows a step of Algorithm 1 of "TACO: Efficient Communication
Compression of Intermediate Tensors for Scalable Tensor-Parallel LLM Training":
block energy (Eq. 6), Adaptive Scale (Eq. 7), orthogonal Hadamard rotation
(Eq. 8), post-rotation scale (Eq. 9), FP8 E4M3 conversion (Eq. 10), and the
inverse (Eqs. 11-13); ``reduce_shards`` is the single local reduction of the
two-shot AllReduce (Section 4.4.2).

Packed format (Section 4.4.2, metadata stored right after the codes): record k occupies
bytes [k*(B+8), (k+1)*(B+8)): B E4M3 codes, then alpha_k and s_k as
little-endian float32.

Ablations (``variant``, ``code`` arguments; default ASH + DS with E4M3):
standard Hadamard + DS (alpha = 1, Section 5.3.1), DS only (alpha = 1, no
rotation, Section 5.2.2), ASH only (s = 1, direct cast, Section 5.2.2); codes
E4M3, E5M2 (Q_max 57344, Section 5.3.2) and INT8 (Q_max 127, round half to
even, Sections 2 and 6).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "taco_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_taco.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

TAU = 1.0
EPS = np.float32(1e-30)
QMAX = 448.0

ASH_DS, HADAMARD_DS, DS_ONLY, ASH_ONLY = 0, 1, 2, 3
E4M3, E5M2, INT8 = 0, 1, 2
VARIANTS = {"ash_ds": ASH_DS, "hadamard_ds": HADAMARD_DS, "ds_only": DS_ONLY, "ash_only": ASH_ONLY}
CODES = {"e4m3": E4M3, "e5m2": E5M2, "int8": INT8}
CODE_QMAX = {E4M3: 448.0, E5M2: 57344.0, INT8: 127.0}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``taco_oracle.c`` into ``liboracle_taco.so`` (gcc) and return its path."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    c_u8p = ctypes.POINTER(ctypes.c_uint8)
    c_u16p = ctypes.POINTER(ctypes.c_uint16)
    c_f32p = ctypes.POINTER(ctypes.c_float)
    c_f64p = ctypes.POINTER(ctypes.c_double)
    i64, i32 = ctypes.c_int64, ctypes.c_int
    sig = {
        "taco_oracle_packed_bytes": (i64, [i64, i32]),
        "taco_oracle_compress_bf16_ex": (i32, [c_u16p, i64, i32, i32, i32, c_u8p]),
        "taco_oracle_compress_f32_ex": (i32, [c_f32p, i64, i32, i32, i32, c_u8p]),
        "taco_oracle_decompress_f32_ex": (i32, [c_u8p, i64, i32, i32, i32, c_f32p]),
        "taco_oracle_decompress_bf16_ex": (i32, [c_u8p, i64, i32, i32, i32, c_u16p]),
        "taco_oracle_reduce_shards_ex": (i32, [ctypes.POINTER(c_u8p), i32, i64, i32, i32, i32, c_u8p]),
        "taco_oracle_code_encode_array": (None, [i32, c_f32p, i64, c_u8p]),
        "taco_oracle_code_encode_bits": (None, [i32, ctypes.c_uint32, i64, c_u8p]),
        "taco_oracle_code_value_array": (None, [i32, c_u8p, i64, c_f64p]),
        "taco_oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "taco_oracle_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
        "taco_oracle_e4m3_encode_array": (None, [c_f32p, i64, c_u8p]),
        "taco_oracle_e4m3_encode_bits": (None, [ctypes.c_uint32, i64, c_u8p]),
        "taco_oracle_e4m3_value_array": (None, [c_u8p, i64, c_f64p]),
        "taco_oracle_bf16_round_array": (None, [c_f32p, i64, c_u16p]),
        "taco_oracle_fwht": (None, [c_f32p, i32]),
        "taco_oracle_fwht_rows": (None, [c_f32p, i64, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def packed_bytes(n: int, block: int) -> int:
    return int(_load().taco_oracle_packed_bytes(n, block))


def compress(x_bf16: np.ndarray, block: int, variant: int = ASH_DS, code: int = E4M3) -> np.ndarray:
    """Algorithm 1 sender (Eqs. 5-10) on a bf16 tensor given as uint16 bit patterns.

    Returns the packed records as a flat uint8 array of (n/B)*(B+8) bytes.
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1)
    out = np.empty(max(packed_bytes(x.size, block), 0), dtype=np.uint8)
    _check(_load().taco_oracle_compress_bf16_ex(_ptr(x, ctypes.c_uint16), x.size, block, variant, code,
                                                _ptr(out, ctypes.c_uint8)), "compress")
    return out


def compress_f32(x: np.ndarray, block: int, variant: int = ASH_DS, code: int = E4M3) -> np.ndarray:
    """Algorithm 1 sender on a float32 tensor (used for the re-compression of a sum)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(max(packed_bytes(x.size, block), 0), dtype=np.uint8)
    _check(_load().taco_oracle_compress_f32_ex(_ptr(x, ctypes.c_float), x.size, block, variant, code,
                                               _ptr(out, ctypes.c_uint8)), "compress_f32")
    return out


def decompress_f32(packed: np.ndarray, n: int, block: int, variant: int = ASH_DS, code: int = E4M3) -> np.ndarray:
    """Algorithm 1 receiver (Eqs. 11-13) returning G' in float32."""
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(n, dtype=np.float32)
    _check(_load().taco_oracle_decompress_f32_ex(_ptr(p, ctypes.c_uint8), n, block, variant, code,
                                                 _ptr(out, ctypes.c_float)), "decompress_f32")
    return out


def decompress(packed: np.ndarray, n: int, block: int, variant: int = ASH_DS, code: int = E4M3) -> np.ndarray:
    """Algorithm 1 receiver returning the bf16 tensor as uint16 bit patterns (RNE)."""
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(n, dtype=np.uint16)
    _check(_load().taco_oracle_decompress_bf16_ex(_ptr(p, ctypes.c_uint8), n, block, variant, code,
                                                  _ptr(out, ctypes.c_uint16)), "decompress")
    return out


def reduce_shards(shards, n: int, block: int, variant: int = ASH_DS, code: int = E4M3) -> np.ndarray:
    """Decode P packed shards to float32, sum them in shard order, compress the sum once."""
    arrs = [np.ascontiguousarray(s, dtype=np.uint8).reshape(-1) for s in shards]
    ptrs = (ctypes.POINTER(ctypes.c_uint8) * len(arrs))(*[_ptr(a, ctypes.c_uint8) for a in arrs])
    out = np.empty(max(packed_bytes(n, block), 0), dtype=np.uint8)
    _check(_load().taco_oracle_reduce_shards_ex(ptrs, len(arrs), n, block, variant, code,
                                                _ptr(out, ctypes.c_uint8)), "reduce_shards")
    return out


def code_encode(code: int, u: np.ndarray) -> np.ndarray:
    """The code format's conversion of float32 values (E4M3 / E5M2 / INT8 bytes)."""
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(-1)
    out = np.empty(u.size, dtype=np.uint8)
    _load().taco_oracle_code_encode_array(code, _ptr(u, ctypes.c_float), u.size, _ptr(out, ctypes.c_uint8))
    return out


def code_encode_bits(code: int, first: int, count: int, out: np.ndarray = None) -> np.ndarray:
    """Codes of the float32 values with bit patterns first .. first + count - 1
    (modulo 2^32), written into `out` (uint8, count elements) if given."""
    if out is None:
        out = np.empty(count, dtype=np.uint8)
    assert out.dtype == np.uint8 and out.size == count and out.flags.c_contiguous
    _load().taco_oracle_code_encode_bits(code, first & 0xFFFFFFFF, count, _ptr(out, ctypes.c_uint8))
    return out


def code_value(code: int, codes: np.ndarray) -> np.ndarray:
    """The float64 value of each code byte of the given format."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    _load().taco_oracle_code_value_array(code, _ptr(c, ctypes.c_uint8), c.size, _ptr(out, ctypes.c_double))
    return out


def e4m3_encode(u: np.ndarray) -> np.ndarray:
    """Cvt_FP8 (Eq. 10) element-wise on float32 values."""
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(-1)
    out = np.empty(u.size, dtype=np.uint8)
    _load().taco_oracle_e4m3_encode_array(_ptr(u, ctypes.c_float), u.size, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_encode_bits(first: int, count: int) -> np.ndarray:
    """Cvt_FP8 of the float32 bit patterns first .. first+count-1."""
    out = np.empty(count, dtype=np.uint8)
    _load().taco_oracle_e4m3_encode_bits(first, count, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """Cvt_FP32 (Eq. 11) element-wise: the float64 value of each E4M3 code."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    _load().taco_oracle_e4m3_value_array(_ptr(c, ctypes.c_uint8), c.size, _ptr(out, ctypes.c_double))
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(x.size, dtype=np.uint16)
    _load().taco_oracle_bf16_round_array(_ptr(x, ctypes.c_float), x.size, _ptr(out, ctypes.c_uint16))
    return out


def fwht(v: np.ndarray, block: int) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of each length-B row (float32, in a copy)."""
    a = np.array(v, dtype=np.float32, copy=True).reshape(-1)
    if a.size % block:
        raise ValueError("size not a multiple of the block")
    _load().taco_oracle_fwht_rows(_ptr(a, ctypes.c_float), a.size // block, block)
    return a.reshape(np.shape(v))


def split_records(packed: np.ndarray, block: int):
    """View packed bytes as (codes [M, B] uint8, alpha [M] float32, s [M] float32)."""
    rec = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1, block + 8)
    codes = rec[:, :block]
    alpha = rec[:, block:block + 4].copy().view("<f4").reshape(-1)
    s = rec[:, block + 4:block + 8].copy().view("<f4").reshape(-1)
    return codes, alpha, s
