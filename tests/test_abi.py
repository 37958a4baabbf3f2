"""The C-ABI library loads without a GPU and exports every entry point that
include/taco.h declares; host-side validation needs no device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"TACO_API\s+[\w\s\*]+?\b(taco_\w+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def lib():
    from fp8_compression_tensor_gb300 import build
    build.build()
    import fp8_compression_tensor_gb300 as t
    return t.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"taco_compress", "taco_decompress", "taco_reduce_shards", "taco_compressed_bytes"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_host_side_queries(lib):
    import fp8_compression_tensor_gb300 as t
    assert lib.taco_abi_version() == 2
    assert t.compressed_bytes(8192, 4096, 128) == 8192 * 4096 // 128 * 136
    assert t.compressed_bytes(0, 4096, 64) == 0
    assert lib.taco_compressed_bytes(16, 100, 64) == -1
    assert lib.taco_compressed_bytes(16, 128, 32) == 16 * 128 // 32 * 40
    assert lib.taco_compressed_bytes(16, 1024, 512) == 16 * 1024 // 512 * 520
    assert lib.taco_compressed_bytes(16, 128, 96) == -1
    assert lib.taco_compressed_bytes(16, 512, 1024) == -1
    assert lib.taco_compressed_bytes(-1, 128, 128) == -1
    assert lib.taco_compressed_bytes(1 << 40, 1 << 40, 128) == -1
    for s in range(10):
        assert lib.taco_status_string(s)
    # Argument errors are found before any CUDA call.
    assert lib.taco_compress(None, 4, 100, 64, None, None) == 2
    assert lib.taco_compress(None, 4, 128, 96, None, None) == 3
    assert lib.taco_compress(None, 4, 128, 128, None, None) == 1
    assert lib.taco_compress(16, 4, 128, 128, 2, None) == 4
    assert lib.taco_compress(0, 0, 128, 128, 0, None) == 0
    # Blocks 64-512 address the tensor with 32-bit row coordinates (rows of
    # min(B, 128) elements); block 32 has no such limit.
    for fn in (lib.taco_compress, lib.taco_decompress):
        assert fn(None, 1 << 31, 64, 64, None, None) == 2
        assert fn(None, (1 << 31) - 1, 64, 64, None, None) == 1
        assert fn(None, 1 << 30, 512, 256, None, None) == 2
        assert fn(None, (1 << 30) - 1, 256, 256, None, None) == 1
        assert fn(None, 1 << 31, 64, 32, None, None) == 1
    ptrs = (ctypes.c_void_p * 1)(16)
    assert lib.taco_reduce_shards(ptrs, 0, 4, 128, 128, 32, None) == 5
    assert lib.taco_reduce_shards(ptrs, 17, 4, 128, 128, 32, None) == 5


def test_options_validated_on_host(lib):
    """The _ex calls check their options before anything else."""
    from fp8_compression_tensor_gb300._binding import _Options
    optp = ctypes.POINTER(_Options)
    for fn in (lib.taco_compress_ex, lib.taco_decompress_ex):
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, optp, ctypes.c_void_p, ctypes.c_void_p]
        assert fn(None, 4, 128, None, None, None) == 9
        assert fn(None, 4, 128, ctypes.byref(_Options(128, 4, 0)), None, None) == 9
        assert fn(None, 4, 128, ctypes.byref(_Options(128, 0, 3)), None, None) == 9
        assert fn(None, 4, 128, ctypes.byref(_Options(128, -1, 0)), None, None) == 9
        assert fn(None, 4, 128, ctypes.byref(_Options(96, 1, 1)), None, None) == 3
        assert fn(None, 4, 100, ctypes.byref(_Options(64, 2, 2)), None, None) == 2
        assert fn(None, 4, 128, ctypes.byref(_Options(128, 3, 1)), None, None) == 1
        assert fn(0, 0, 128, ctypes.byref(_Options(128, 1, 2)), 0, None) == 0
    lib.taco_reduce_shards_ex.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int64, optp, ctypes.c_void_p, ctypes.c_void_p]
    ptrs = (ctypes.c_void_p * 1)(16)
    assert lib.taco_reduce_shards_ex(ptrs, 1, 4, 128, None, 32, None) == 9
    assert lib.taco_reduce_shards_ex(ptrs, 0, 4, 128, ctypes.byref(_Options(128, 1, 1)), 32, None) == 5


def test_binding_refuses_cpu_tensors():
    import torch
    import fp8_compression_tensor_gb300 as t
    with pytest.raises(TypeError):
        t.compress(torch.zeros(4, 128, dtype=torch.bfloat16), 128)


def test_encode_selftest_validated_on_host(lib):
    """taco_selftest_encode_bits checks its arguments before any device call."""
    fn = lib.taco_selftest_encode_bits
    assert fn(3, 0, 16, 16, None) == 9            # unknown code format
    assert fn(-1, 0, 16, 16, None) == 9
    assert fn(0, 0, 6, 16, None) == 2             # count not a multiple of 4
    assert fn(0, 2, 16, 16, None) == 2            # first not a multiple of 4
    assert fn(0, 0, (1 << 32) + 4, 16, None) == 2  # more than every pattern
    assert fn(0, 0, -4, 16, None) == 2
    assert fn(1, 0, 0, None, None) == 0           # nothing to do
    assert fn(1, 0, 16, None, None) == 1          # null output
    assert fn(2, 0, 16, 8, None) == 4             # misaligned output

