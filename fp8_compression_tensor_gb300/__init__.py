"""GB300 (sm_103a) implementation of TACO's fused FP8 compression of
tensor-parallel intermediate tensors ("TACO: Efficient Communication
Compression of Intermediate Tensors for Scalable Tensor-Parallel LLM
Training", Algorithm 1; Sections 4.2-4.4).

    packed = compress(x_bf16, block=128)            # Eqs. 5-10, one fused kernel
    y = decompress(packed, rows, hidden, block=128)  # Eqs. 11-13, one fused kernel
    r = reduce_shards([p0, ..., pP-1], rows, hidden, block=128)  # two-shot local reduction

Every call also takes variant= ("ash_ds", "hadamard_ds", "ds_only",
"ash_only") and code= ("e4m3", "e5m2", "int8") for the paper's ablations.

The kernels live in libtaco_gb300.so (C ABI: include/taco.h); this package
only marshals arguments.  Build the library with
`python -m fp8_compression_tensor_gb300.build`.
"""
from ._binding import (CODES, LIBRARY_PATH, MAX_SHARDS, STATUS, SUPPORTED_BLOCKS, VARIANTS,  # noqa: F401
                       TacoError, compress, compressed_bytes, decompress, device_status, load_library, raw_call,
                       reduce_shards, selftest_encode_bits)

__all__ = ["compress", "decompress", "reduce_shards", "compressed_bytes", "device_status", "load_library",
           "TacoError", "LIBRARY_PATH", "MAX_SHARDS", "SUPPORTED_BLOCKS", "STATUS", "VARIANTS", "CODES",
           "raw_call", "selftest_encode_bits"]
