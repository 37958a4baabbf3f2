// taco_selftest.cu -- the wait-timeout self-test behind
// taco_selftest_wait_timeout(): one CTA waits, with a short limit, on an
// mbarrier that nothing ever completes, takes the same give-up path as every
// kernel's bounded waits (set a fault bit, return) and exits.  It exercises
// the device fault flags end to end without faulting, trapping or hanging the
// GPU.
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

}  // namespace

cudaError_t launch_wait_selftest(uint32_t *fault, uint64_t limit_ns, cudaStream_t stream)
{
    taco_wait_selftest_kernel<<<1, 32, 0, stream>>>(fault, limit_ns);
    return cudaGetLastError();
}

}  // namespace taco
