// taco_kernels.h -- host-side view of the TACO kernels (internal to the library).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace taco {

// Launch facts of one kernel instantiation.
struct KernelInfo {
    void *fn = nullptr;     // kernel entry (for attributes and occupancy queries)
    size_t smem = 0;        // dynamic shared memory per CTA
    int threads = 0;        // threads per CTA
    int tile_blocks = 0;    // blocks per CTA tile
    int warps = 0;          // warps per CTA
};

#ifndef TACO_PDL
#define TACO_PDL 1
#endif

// Launches `fn` with programmatic stream serialisation (when TACO_PDL): the
// kernel may be scheduled while the previous kernel in the stream finishes;
// the kernels order their memory accesses with griddepcontrol.wait.
inline cudaError_t launch_kernel(const void *fn, int grid, int threads, size_t smem, cudaStream_t stream, void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = TACO_PDL ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Compression scheme: the method (ASH + DS with E4M3 codes) or one of the
// paper's ablations.  Variants: 0 ASH + DS, 1 standard Hadamard + DS
// (alpha = 1), 2 DS only (alpha = 1, no rotation), 3 ASH only (s = 1).
// Codes: 0 E4M3 (Q_max 448), 1 E5M2 (57344), 2 INT8 (127, ties to even).
struct Scheme {
    int variant;
    int code;
};

KernelInfo compress_kernel_info(int block, int variant, int code);   // DS only, and INT8 codes, have their own kernels
KernelInfo decompress_kernel_info(int block, int code);   // code 2 (INT8) has its own kernel
KernelInfo reduce_kernel_info(int block, int code, int num_shards);

// `tmap` points to a CUtensorMap of x viewed as [nblocks, block] bf16, box
// {64, 128}, 128-byte swizzle.
cudaError_t launch_compress(int block, Scheme scheme, const void *tmap, void *packed, int64_t nblocks, uint32_t *fault,
                            int grid, cudaStream_t stream);
// `tmap_y` points to a CUtensorMap of y viewed as [nblocks, block] bf16, box
// {64, tile_blocks}, 128-byte swizzle.
cudaError_t launch_decompress(int block, Scheme scheme, const void *tmap_y, const void *packed, int64_t nblocks,
                              uint32_t *fault, int grid, cudaStream_t stream);

// CUDA-core codec for block 32 (a lane per block); fn == nullptr otherwise.
// tile_blocks = blocks per CTA.
KernelInfo warp_codec_info(int block, bool compress, int code);   // INT8 compress has its own kernel
cudaError_t launch_warp_compress(int block, Scheme scheme, const void *x, void *packed, int64_t nblocks, int grid,
                                 cudaStream_t stream);
cudaError_t launch_warp_decompress(int block, Scheme scheme, const void *packed, void *y, int64_t nblocks, int grid,
                                   cudaStream_t stream);

// One CTA whose wait on a barrier nothing completes gives up after limit_ns
// and sets the self-test fault bit.
cudaError_t launch_wait_selftest(uint32_t *fault, uint64_t limit_ns, cudaStream_t stream);

constexpr int kMaxShards = 16;

struct ReduceArgs {
    const uint8_t *shards[kMaxShards];
    uint8_t *out;
    int64_t nblocks;
    int num_shards;
    int variant;    // Scheme::variant (the code format selects the kernel)
};

// One CTA per tile of KernelInfo::tile_blocks blocks (tiles of CTAs that have
// not started are taken over by running ones).
cudaError_t launch_reduce(int block, int code, const ReduceArgs &args, uint32_t *fault, int grid, cudaStream_t stream);

}  // namespace taco
