// taco_tcgen05.cuh -- inline-PTX wrappers for the Blackwell tensor-core path
// (sm_100 family): tensor-memory allocation, tcgen05.mma with shared-memory
// matrix descriptors, tcgen05.commit to an mbarrier, tcgen05.ld, 2-D tiled
// TMA loads, named barriers and single-thread bounded mbarrier waits.
#pragma once

#include <cstdint>

#include "taco_device.cuh"

namespace taco {

// ---------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------

// Allocates `ncols` (a power of two >= 32) TMEM columns for this CTA and
// writes the base address to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees what tmem_alloc returned.  Whole warp (the allocating one).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-wide:
// lane i of the warp reads TMEM lane (taddr >> 16) + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Orders every use of r after the tmem_ld_wait before it (the registers a
// tcgen05.ld writes are valid only after the wait, which the compiler cannot
// see).
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Writes 32 consecutive 32-bit TMEM columns of this thread's lane (warp-wide,
// the layout of tmem_ld32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// MMA
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes, 16-byte units XOR-swizzled by
// (row % 8), 8-row groups 1024 bytes apart.  `addr` is the shared-memory
// address of the first row (1024-byte aligned region, plus a multiple of 32
// bytes to step along K inside the 128-byte row).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);          // start address
    d |= static_cast<uint64_t>(1u) << 16;                       // leading byte offset (unused here)
    d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;   // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1u) << 46;                       // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2u) << 61;                       // swizzle: 128 bytes
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16 with BF16 A and B (both
// K-major), FP32 accumulation, shape M x N.
__host__ __device__ constexpr uint32_t mma_idesc_bf16_f32(int M, int N)
{
    return (1u << 4)                                   // D format: F32
           | (1u << 7)                                 // A format: BF16
           | (1u << 10)                                // B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 with E4M3 A and B (both
// K-major), FP32 accumulation, shape M x N.
__host__ __device__ constexpr uint32_t mma_idesc_e4m3_f32(int M, int N)
{
    return (1u << 4)                                   // D format: F32
           | (0u << 7)                                 // A format: E4M3
           | (0u << 10)                                // B format: E4M3
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor of tcgen05.mma.kind::f16 with F16 A and B (format 0).
__host__ __device__ constexpr uint32_t mma_idesc_f16_f32(int M, int N)
{
    return (1u << 4)                                   // D format: F32
           | (0u << 7)                                 // A format: F16
           | (0u << 10)                                // B format: F16
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Same with E5M2 A and B (format 1 of .kind::f8f6f4).
__host__ __device__ constexpr uint32_t mma_idesc_e5m2_f32(int M, int N)
{
    return (1u << 4)                                   // D format: F32
           | (1u << 7)                                 // A format: E5M2
           | (1u << 10)                                // B format: E5M2
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}


// D[tmem] = A * B^T (+ D if accumulate): A is M x K, B is N x K, both from
// shared-memory descriptors, 16-bit operands (BF16 or F16 per the
// instruction descriptor, K = 16).  Issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with 8-bit operands (.kind::f8f6f4): K = 32 per instruction.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier at `bar` receives one arrival once every tcgen05.mma this
// thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Cluster launch control (dynamic tile scheduling)
// ---------------------------------------------------------------------------

// Asks the hardware to cancel one CTA of this grid that has not started yet;
// the 16-byte response lands at `result_addr` (16-byte aligned shared memory)
// and completes 16 transaction bytes on `bar` (the caller arrives on `bar`
// with expect_tx(16) first).  No request may be issued once a failed
// response has been observed.
__device__ __forceinline__ void clc_try_cancel(uint32_t result_addr, uint32_t bar)
{
    asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
                 ::"r"(result_addr), "r"(bar)
                 : "memory");
}

// Reads a response: the x index of the cancelled CTA (whose work the caller
// now does), or -1 if no CTA was left to cancel.
__device__ __forceinline__ int64_t clc_response_ctaid_x(uint32_t result_addr)
{
    uint32_t ok, x = 0;
    // The cancelled CTA's index is read only from a successful response.
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "+r"(x)
        : "r"(result_addr)
        : "memory");
    return ok ? static_cast<int64_t>(x) : -1;
}

// ---------------------------------------------------------------------------
// TMA, barriers
// ---------------------------------------------------------------------------

// 2-D tiled bulk tensor load of the box at (x, y) into shared memory; the
// bytes complete on `bar`.  x (innermost, in elements) must keep x*elem_size
// a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Hint: fetch the box at (x, y) from HBM into L2 (same coordinate rules as
// tma_load_2d; see bulk_prefetch_l2 for why it may precede the dependency wait).
__device__ __forceinline__ void tma_prefetch_2d(const void *tmap, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y)
                 : "memory");
}

// 2-D tiled bulk tensor store of a shared-memory box to (x, y); elements
// outside the tensor are not written.  Tracked by bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const void *tmap, int32_t x, int32_t y, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Single-thread bounded wait for phase `parity` of `bar` (limit_ns, by
// default kWaitLimitNs); sets `fault_bit` and returns false on a timeout.
__device__ __forceinline__ bool mbar_wait_bounded_thread(uint32_t bar, uint32_t parity, uint32_t *fault,
                                                         uint32_t fault_bit, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(fault, fault_bit);
            return false;
        }
    }
    return true;
}

}  // namespace taco
