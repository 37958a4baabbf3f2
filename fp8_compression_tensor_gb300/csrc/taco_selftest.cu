// taco_selftest.cu -- self-tests of the library's device code.
//
// taco_selftest_wait_timeout(): one CTA waits, with a short limit, on an
// mbarrier that nothing ever completes, takes the same give-up path as every
// kernel's bounded waits (set a fault bit, return) and exits.  It exercises
// the device fault flags end to end without faulting, trapping or hanging the
// GPU.
//
// taco_selftest_encode_bits(): the code conversion every kernel uses
// (encode4: E4M3 and E5M2 by the hardware's saturating conversions, INT8 by
// round-half-even integer conversion) applied to a range of float32 bit
// patterns, so that it can be compared with an independent encoder over
// every input.
#include "taco_device.cuh"
#include "taco_kernels.h"
#include "taco_tcgen05.cuh"

namespace taco {
namespace {

__global__ void taco_wait_selftest_kernel(uint32_t *fault, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        // No thread arrives on the barrier: its phase 0 never completes.
        mbar_wait_bounded_thread(b, 0, fault, kFaultSelfTest, limit_ns);
    }
}

// codes[i] = encode(code, float with bits first + i); four per thread.
__global__ void taco_encode_selftest_kernel(int code, uint32_t first, int64_t quads, uint32_t *codes)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < quads;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint32_t b = first + static_cast<uint32_t>(4 * i);   // modulo 2^32
        codes[i] = encode4(code, __uint_as_float(b), __uint_as_float(b + 1u), __uint_as_float(b + 2u),
                           __uint_as_float(b + 3u));
    }
}

}  // namespace

cudaError_t launch_encode_selftest(int code, uint32_t first, int64_t count, void *codes, int grid,
                                   cudaStream_t stream)
{
    taco_encode_selftest_kernel<<<grid, 256, 0, stream>>>(code, first, count / 4, static_cast<uint32_t *>(codes));
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t *fault, uint64_t limit_ns, cudaStream_t stream)
{
    taco_wait_selftest_kernel<<<1, 32, 0, stream>>>(fault, limit_ns);
    return cudaGetLastError();
}

}  // namespace taco
