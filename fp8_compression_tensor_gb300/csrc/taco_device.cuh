// taco_device.cuh -- device-side building blocks shared by the TACO kernels:
// the fixed constants, inline-PTX wrappers for mbarriers and bulk copies,
// E4M3 / bf16 conversions, packed FP32x2 arithmetic and the bounded wait.
//
// Method: "TACO: Efficient Communication Compression of Intermediate Tensors
// for Scalable Tensor-Parallel LLM Training", Algorithm 1, Eqs. (6)-(13).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace taco {

// Constants the paper leaves open (Eqs. 6, 7, 9): target RMS tau, eps inside
// the root, largest finite E4M3 value.
constexpr float kTau = 1.0f;
constexpr float kEps = 1e-30f;
constexpr float kQmax = 448.0f;

// Blocks at the bottom of the binary32 range (the near-zero region where the
// Adaptive Scale makes alpha ~ 1e15).  The kernels work on unscaled values
// (the rotation y = H G, or a shard's factor s / alpha), which there sit near
// or inside the subnormal range: Q_max / max|y| overflows once max|y| <
// Q_max / FLT_MAX (2^-119.2 for E4M3, 2^-112.2 for E5M2), and a subnormal
// factor keeps only a few significant bits.  Below kTinyValue such a value is
// multiplied by kTinyUp = 2^64 first (exact) and the result by kTinyDown =
// 2^-64 at the end, which gives the same roundings as the unscaled formula
// would in a binary32 without overflow or underflow.
constexpr float kTinyValue = 0x1p-100f;
// The shard reduce detects such blocks by their sum: below 2^-80 every
// factor s_p / alpha_p may lie in that range (sum_p 448 s_p / alpha_p bounds it).
constexpr float kTinySum = 0x1p-80f;
constexpr float kTinyUp = 0x1p64f;
constexpr float kTinyDown = 0x1p-64f;
// Smallest divisor for which div2_by (reciprocal and one correction) is used.
constexpr float kDivFastMin = 0x1p-100f;

// Fault flag bits written when a kernel gives up waiting.
constexpr uint32_t kFaultCompress = 1u;
constexpr uint32_t kFaultDecompress = 2u;
constexpr uint32_t kFaultReduce = 4u;
constexpr uint32_t kFaultSelfTest = 8u;   // the wait-timeout self-test (taco_selftest_wait_timeout)

// A wait on the copy engine gives up after this long (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Shared memory, mbarriers and bulk copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses with later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

#ifndef TACO_WAIT_HINT_NS
#define TACO_WAIT_HINT_NS 1000000
#endif

// Tests phase `parity` of the barrier; if it is not complete, the thread may
// be suspended (instead of spinning) until it completes or about
// TACO_WAIT_HINT_NS nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(TACO_WAIT_HINT_NS)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier, for at most kWaitLimitNs.  The
// outcome is the same for every lane of the warp.  On a timeout the fault bit
// is set and false is returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t *fault,
                                                  uint32_t fault_bit)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_timer_ns();
        while (!(ok = mbar_try_wait(bar, parity))) {
            if (global_timer_ns() - t0 > kWaitLimitNs)
                break;
        }
    }
    ok = __all_sync(kFullMask, ok);
    if (!ok && (threadIdx.x & 31) == 0)
        atomicOr(fault, fault_bit);
    return ok;
}

// Bulk copy global -> shared (size a multiple of 16, both addresses 16-byte
// aligned); completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Hint: fetch [src, src + bytes) from HBM into L2 (size a multiple of 16,
// src 16-byte aligned).  Nothing reaches the SM and L2 is the device's point
// of coherence for global memory, so a prefetch can never make a later load
// return stale data: a kernel may issue it before grid_dependency_wait() to
// overlap the first DRAM round trip with the previous kernel's tail.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Number of SMs of the device (an upper bound on the SM ids).
__device__ __forceinline__ uint32_t num_sms()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%nsmid;" : "=r"(n));
    return n;
}

// Bulk copy shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// At most N of this thread's bulk groups may still be reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// At most N of this thread's bulk groups may still be in flight.
template <int N>
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream is still
// running; grid_dependency_wait() returns once that kernel has completed and
// its memory operations are visible (at once for an ordinary launch), so every
// thread calls it before its first global-memory access.
// grid_launch_dependents() lets the next kernel in the stream be scheduled
// (on the SM resources this grid frees) before this one has finished.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// CTA-wide barrier over all threads, counted thread by thread (the
// non-aligned form): lanes of one warp that took different paths (a
// single-lane producer or issuer) may arrive separately.  The aligned form
// behind __syncthreads() expects whole converged warps and may release early
// when a warp arrives in pieces.
__device__ __forceinline__ void cta_barrier()
{
    asm volatile("barrier.sync 0;" ::: "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b)
{
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// ---------------------------------------------------------------------------
// Packed FP32x2 arithmetic (one instruction for two lanes of data)
// ---------------------------------------------------------------------------

// Packed add written as PTX (one instruction for two lanes of data).
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// y / s rounded to nearest for the two values of y, given rcp = 1/s
// correctly rounded (__frcp_rn): the quotient q = y * rcp is corrected once,
// q + (y - q s) * rcp, the residual y - q s being exact in a fused
// multiply-add.  This gives the correctly rounded quotient (the classic
// correction step for a correctly rounded reciprocal; the test suite checks it
// against exact rational division on random and on exact quotients).  Valid for
// a normal s with 2^-100 <= s < 2^100; callers divide exactly otherwise.
__device__ __forceinline__ float2 div2_by(float2 y, float s, float rcp)
{
    const float2 r2 = make_float2(rcp, rcp), s2 = make_float2(s, s);
    const float2 q = __fmul2_rn(y, r2);
    const float2 e = __ffma2_rn(make_float2(-q.x, -q.y), s2, y);
    return __ffma2_rn(e, r2, q);
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// Cvt_FP8 (Eq. 10) of two floats: round to nearest even, saturate to +-448.
// Returns 16 bits: `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint32_t e4m3x2_from_float2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Same conversion to OCP E5M2 (round to nearest even, saturating to +-57344).
__device__ __forceinline__ uint32_t e5m2x2_from_float2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Largest code magnitude of a code format (0 E4M3, 1 E5M2, 2 INT8).
__device__ __forceinline__ float code_qmax(int code)
{
    return code == 0 ? 448.0f : code == 1 ? 57344.0f : 127.0f;
}

// INT8 codes of four values (first in the low byte), rounded to the nearest
// integer, ties to even, for |u| < 2^22: u + 1.5 * 2^23 lies in [2^23, 2^24),
// where FP32 values are spaced by 1, so the FP32 add rounds u to an integer
// (nearest, ties to even) and the low byte of the sum's bits is that integer
// modulo 256, its two's-complement byte.
constexpr float kInt8Magic = 12582912.0f;   // 1.5 * 2^23
__device__ __forceinline__ uint32_t int8x4_from_float(float a, float b, float c, float d)
{
    const float2 m = make_float2(kInt8Magic, kInt8Magic);
    const float2 x = add2(make_float2(a, b), m), y = add2(make_float2(c, d), m);
    const uint32_t lo = __byte_perm(__float_as_uint(x.x), __float_as_uint(x.y), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(y.x), __float_as_uint(y.y), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// Values of four INT8 codes (exact): the byte v ^ 0x80 = v + 128 under the
// exponent byte 0x4B is the FP32 value 2^23 + v + 128, and subtracting
// 2^23 + 128 is exact.
__device__ __forceinline__ void int8x4_to_float(uint32_t x, float2 &q0, float2 &q1)
{
    const uint32_t u = x ^ 0x80808080u;
    const float2 off = make_float2(-8388736.0f, -8388736.0f);   // -(2^23 + 128)
    q0 = add2(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                          __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))),
              off);
    q1 = add2(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                          __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))),
              off);
}

// Codes of four values, first value in the low byte.  INT8 rounds to the
// nearest integer, ties to even; the callers keep |u| <= 127 (u = Q_max y /
// max|y| rounds to at most 127, and a direct cast has |u| <= sqrt(B) <= sqrt(512),
// about 22.6).
__device__ __forceinline__ uint32_t encode4(int code, float a, float b, float c, float d)
{
    if (code == 0)
        return e4m3x2_from_float2(a, b) | (e4m3x2_from_float2(c, d) << 16);
    if (code == 1)
        return e5m2x2_from_float2(a, b) | (e5m2x2_from_float2(c, d) << 16);
    return int8x4_from_float(a, b, c, d);
}

// Codes of the four products ab.x k, ab.y k, cd.x k, cd.y k (first in the low
// byte), each product rounded to binary32 before the conversion.  INT8 takes
// scalar products: a packed multiply followed by the packed rounding add of
// int8x4_from_float came out fused into one fused multiply-add, which rounds
// the exact product to an integer (63.4999993 -> 63 where the binary32
// product is 63.5 -> 64).  The FP8 conversions read the packed products.
__device__ __forceinline__ uint32_t encode4_scaled(int code, float2 ab, float2 cd, float k)
{
    if (code == 2)
        return int8x4_from_float(__fmul_rn(ab.x, k), __fmul_rn(ab.y, k), __fmul_rn(cd.x, k), __fmul_rn(cd.y, k));
    const float2 k2 = make_float2(k, k);
    const float2 u0 = mul2(ab, k2), u1 = mul2(cd, k2);
    return encode4(code, u0.x, u0.y, u1.x, u1.y);
}

// Cvt_FP32 (Eq. 11) of the two E4M3 codes in the low 16 bits of `pair`
// (exact): low byte -> .x, high byte -> .y.
// The two f16 values of a word as floats (exact), low half first.
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h2)
{
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(pair)));
    return f16x2_to_float2(h2);
}

// The two E5M2 codes in the low 16 bits of `pair` as floats (exact).
__device__ __forceinline__ float2 e5m2x2_to_float2(uint32_t pair)
{
    // An E5M2 code is the high byte of the f16 of the same value.
    return f16x2_to_float2(__byte_perm(pair, 0u, 0x1404));
}

// Two floats -> two bf16 (round to nearest even) packed in a word, lo first.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace taco
