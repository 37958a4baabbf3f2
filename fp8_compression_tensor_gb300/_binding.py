"""ctypes binding of libtaco_gb300.so (the C ABI in include/taco.h).

Argument marshalling only: every step of compress / decompress / reduce runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.
There is no CPU fallback: if the library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_PKG, "libtaco_gb300.so")

STATUS = {
    0: "TACO_OK",
    1: "TACO_ERR_NULL_POINTER",
    2: "TACO_ERR_BAD_SHAPE",
    3: "TACO_ERR_UNSUPPORTED_BLOCK",
    4: "TACO_ERR_MISALIGNED",
    5: "TACO_ERR_BAD_SHARDS",
    6: "TACO_ERR_OVERLAP",
    7: "TACO_ERR_CUDA",
    8: "TACO_ERR_DEVICE_FAULT",
    9: "TACO_ERR_BAD_OPTIONS",
}
MAX_SHARDS = 16
SUPPORTED_BLOCKS = (32, 64, 128, 256, 512)
# Ablations (taco_variant_t, taco_code_t of include/taco.h).
VARIANTS = {"ash_ds": 0, "hadamard_ds": 1, "ds_only": 2, "ash_only": 3}
CODES = {"e4m3": 0, "e5m2": 1, "int8": 2}


class _Options(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("variant", ctypes.c_int), ("code", ctypes.c_int)]


def _options(block: int, variant, code) -> Optional[_Options]:
    """None for the method itself (ASH + DS, E4M3), else the _ex options."""
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    c = CODES[code] if isinstance(code, str) else int(code)
    if v == 0 and c == 0:
        return None
    return _Options(block, v, c)

_lock = threading.Lock()
_lib = None


class TacoError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {name}{(' ' + detail) if detail else ''}")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("TACO_GB300_LIBRARY") or LIBRARY_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m fp8_compression_tensor_gb300.build`")
        lib = ctypes.CDLL(p)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.taco_compressed_bytes.argtypes = [i64, i64, i32]
        lib.taco_compressed_bytes.restype = i64
        lib.taco_compress.argtypes = [vp, i64, i64, i32, vp, vp]
        lib.taco_compress.restype = i32
        lib.taco_decompress.argtypes = [vp, i64, i64, i32, vp, vp]
        lib.taco_decompress.restype = i32
        lib.taco_reduce_shards.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i32, vp, vp]
        lib.taco_reduce_shards.restype = i32
        optp = ctypes.POINTER(_Options)
        lib.taco_compress_ex.argtypes = [vp, i64, i64, optp, vp, vp]
        lib.taco_compress_ex.restype = i32
        lib.taco_decompress_ex.argtypes = [vp, i64, i64, optp, vp, vp]
        lib.taco_decompress_ex.restype = i32
        lib.taco_reduce_shards_ex.argtypes = [ctypes.POINTER(vp), i32, i64, i64, optp, vp, vp]
        lib.taco_reduce_shards_ex.restype = i32
        lib.taco_selftest_wait_timeout.argtypes = [vp]
        lib.taco_selftest_wait_timeout.restype = i32
        lib.taco_selftest_encode_bits.argtypes = [i32, ctypes.c_uint32, i64, vp, vp]
        lib.taco_selftest_encode_bits.restype = i32
        lib.taco_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.taco_device_status.restype = i32
        lib.taco_status_string.argtypes = [i32]
        lib.taco_status_string.restype = ctypes.c_char_p
        lib.taco_last_cuda_error.argtypes = []
        lib.taco_last_cuda_error.restype = i32
        lib.taco_abi_version.argtypes = []
        lib.taco_abi_version.restype = i32
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        lib = load_library()
        detail = ""
        if rc == 7:
            detail = f"(cudaError {lib.taco_last_cuda_error()})"
        raise TacoError(rc, what, detail)


def _stream_handle(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_cuda_tensor(t: torch.Tensor, dtype: torch.dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def compressed_bytes(rows: int, hidden: int, block: int = 128) -> int:
    """Size in bytes of the packed records of a [rows, hidden] tensor."""
    n = load_library().taco_compressed_bytes(rows, hidden, block)
    if n < 0:
        status = 3 if block not in SUPPORTED_BLOCKS else 2
        raise TacoError(status, "compressed_bytes", f"(rows={rows} hidden={hidden} block={block})")
    return int(n)


def _rows_hidden(x: torch.Tensor):
    if x.dim() == 0:
        raise ValueError("tensor must have at least one dimension")
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    return rows, hidden


def compress(x: torch.Tensor, block: int = 128, out: Optional[torch.Tensor] = None, stream=None,
             variant="ash_ds", code="e4m3") -> torch.Tensor:
    """TACO compression (Algorithm 1 sender side) of a bf16 CUDA tensor, viewed
    as [rows, hidden] with hidden = x.shape[-1].  Returns (or fills) a uint8
    tensor of compressed_bytes(rows, hidden, block) packed bytes.  `variant`
    and `code` select an ablation (VARIANTS, CODES)."""
    _check_cuda_tensor(x, torch.bfloat16, "x")
    rows, hidden = _rows_hidden(x)
    nbytes = compressed_bytes(rows, hidden, block)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    else:
        _check_cuda_tensor(out, torch.uint8, "out")
        if out.numel() != nbytes:
            raise ValueError(f"out must have {nbytes} bytes, has {out.numel()}")
    opt = _options(block, variant, code)
    with torch.cuda.device(x.device):
        if opt is None:
            rc = load_library().taco_compress(x.data_ptr(), rows, hidden, block, out.data_ptr(),
                                              _stream_handle(x.device, stream))
        else:
            rc = load_library().taco_compress_ex(x.data_ptr(), rows, hidden, ctypes.byref(opt), out.data_ptr(),
                                                 _stream_handle(x.device, stream))
    _check(rc, "taco_compress")
    return out


def decompress(packed: torch.Tensor, rows: int, hidden: int, block: int = 128,
               out: Optional[torch.Tensor] = None, stream=None, variant="ash_ds", code="e4m3") -> torch.Tensor:
    """TACO decompression (Algorithm 1 receiver side) of packed records into a
    bf16 [rows, hidden] CUDA tensor."""
    _check_cuda_tensor(packed, torch.uint8, "packed")
    nbytes = compressed_bytes(rows, hidden, block)
    if packed.numel() != nbytes:
        raise ValueError(f"packed must have {nbytes} bytes, has {packed.numel()}")
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=packed.device)
    else:
        _check_cuda_tensor(out, torch.bfloat16, "out")
        if out.numel() != rows * hidden:
            raise ValueError("out has the wrong number of elements")
    opt = _options(block, variant, code)
    with torch.cuda.device(packed.device):
        if opt is None:
            rc = load_library().taco_decompress(packed.data_ptr(), rows, hidden, block, out.data_ptr(),
                                                _stream_handle(packed.device, stream))
        else:
            rc = load_library().taco_decompress_ex(packed.data_ptr(), rows, hidden, ctypes.byref(opt),
                                                   out.data_ptr(), _stream_handle(packed.device, stream))
    _check(rc, "taco_decompress")
    return out


def reduce_shards(shards: Sequence[torch.Tensor], rows: int, hidden: int, block: int = 128,
                  out: Optional[torch.Tensor] = None, stream=None, variant="ash_ds", code="e4m3") -> torch.Tensor:
    """Decode P packed shards of a [rows, hidden] tensor, sum them in FP32 and
    compress the sum once (the local reduction of a two-shot AllReduce)."""
    shards = list(shards)
    if not 1 <= len(shards) <= MAX_SHARDS:
        raise ValueError(f"need 1..{MAX_SHARDS} shards, got {len(shards)}")
    nbytes = compressed_bytes(rows, hidden, block)
    for i, s in enumerate(shards):
        _check_cuda_tensor(s, torch.uint8, f"shards[{i}]")
        if s.numel() != nbytes:
            raise ValueError(f"shards[{i}] must have {nbytes} bytes")
    dev = shards[0].device
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    else:
        _check_cuda_tensor(out, torch.uint8, "out")
        if out.numel() != nbytes:
            raise ValueError(f"out must have {nbytes} bytes")
    ptrs = (ctypes.c_void_p * len(shards))(*[s.data_ptr() for s in shards])
    opt = _options(block, variant, code)
    with torch.cuda.device(dev):
        if opt is None:
            rc = load_library().taco_reduce_shards(ptrs, len(shards), rows, hidden, block, out.data_ptr(),
                                                   _stream_handle(dev, stream))
        else:
            rc = load_library().taco_reduce_shards_ex(ptrs, len(shards), rows, hidden, ctypes.byref(opt),
                                                      out.data_ptr(), _stream_handle(dev, stream))
    _check(rc, "taco_reduce_shards")
    return out


def selftest_encode_bits(code, first: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """Self-test of the kernels' code conversion: fills the uint8 CUDA tensor
    `out` with the codes of the float32 bit patterns first, first + 1, ...
    (taco_selftest_encode_bits)."""
    _check_cuda_tensor(out, torch.uint8, "out")
    c = CODES[code] if isinstance(code, str) else int(code)
    with torch.cuda.device(out.device):
        rc = load_library().taco_selftest_encode_bits(c, first & 0xFFFFFFFF, out.numel(), out.data_ptr(),
                                                      _stream_handle(out.device, stream))
    _check(rc, "taco_selftest_encode_bits")
    return out


def device_status(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device fault flags;
    raises TacoError if a kernel gave up waiting for a copy."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(device):
        rc = load_library().taco_device_status(_stream_handle(device, stream), ctypes.byref(flags))
    if rc == 8:
        raise TacoError(rc, "taco_device_status", f"(flags {flags.value:#x})")
    _check(rc, "taco_device_status")
    return flags.value


def raw_call(name: str, *args) -> int:
    """Calls a C-ABI entry point with raw arguments and returns its status
    (used to exercise argument validation directly)."""
    return getattr(load_library(), name)(*args)
