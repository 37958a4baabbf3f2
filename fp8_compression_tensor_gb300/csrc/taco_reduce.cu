// taco_reduce.cu -- receive-side local reduction of TACO's two-shot compressed
// AllReduce (Section 4.4.2, "one compressed AlltoAll operation followed by a
// single local reduction") for GB300 (sm_103a): P packed shards in local HBM
// are decoded to FP32, summed, and the sum is compressed once.
//
// No rotation is needed.  Shard p decodes to G'_p = R (q_p s_p / alpha_p) with
// R = (1/sqrt B) H_B, and R is symmetric and orthogonal (R R = I).  For the sum
// S = R W with W = sum_p q_p (s_p / alpha_p); compressing S gives
// mean(S^2) = |W|^2 / B, Z = alpha' R S = alpha' W, s' = alpha' max|W| / Q_max and
// codes Cvt_FP8(Q_max W / max|W|).  The kernel computes exactly these, which
// differ from decode-sum-encode with explicit rotations only by FP32 rounding.
//
// Layout.  B/16 consecutive lanes share a block; each lane owns 16 elements,
// i.e. 16 bytes of codes per shard (two 8-byte loads: records are 8-byte
// aligned), so a warp reads whole records.  Energy and maximum are reduced across the block's
// lanes with xor-shuffles (every lane ends with the same bits).
#include "taco_device.cuh"
#include "taco_kernels.h"

namespace taco {
namespace {

#ifndef TACO_REDUCE_PACKED_ADD
#define TACO_REDUCE_PACKED_ADD 1
#endif
#ifndef TACO_REDUCE_THREADS
#define TACO_REDUCE_THREADS 128
#endif
#ifndef TACO_REDUCE_BATCH
#define TACO_REDUCE_BATCH 4
#endif
constexpr int kReduceThreads = TACO_REDUCE_THREADS;
constexpr int kLaneCodes = 16;                  // codes (elements) per lane per shard
constexpr int kBatch = TACO_REDUCE_BATCH;       // shards whose loads are issued together

// 16 code bytes of a record.  Records start at multiples of B + 8 bytes,
// which are only 8-byte aligned, so the bytes come in two 8-byte loads.
__device__ __forceinline__ uint4 ldg_codes16(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.z), "=r"(v.w) : "l"(p + 8));
    return v;
}

__device__ __forceinline__ uint2 ldg_nc_u2(const uint8_t *p)
{
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// w[0..15] += q[0..15] * f for the 16 codes in `c`, each product rounded on its
// own before the add (so that a shard and its negation cancel exactly, as in
// an FP32 sum of decoded shards).
__device__ __forceinline__ void accumulate_shard(float (&w)[kLaneCodes], uint4 c, float f)
{
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float2 q0 = e4m3x2_to_float2(words[k] & 0xffffu);
        const float2 q1 = e4m3x2_to_float2(words[k] >> 16);
#if TACO_REDUCE_PACKED_ADD
        // Scalar products (never contracted), packed sums.
        const float2 t0 = make_float2(__fmul_rn(q0.x, f), __fmul_rn(q0.y, f));
        const float2 t1 = make_float2(__fmul_rn(q1.x, f), __fmul_rn(q1.y, f));
        const float2 s0 = add2(make_float2(w[4 * k + 0], w[4 * k + 1]), t0);
        const float2 s1 = add2(make_float2(w[4 * k + 2], w[4 * k + 3]), t1);
        w[4 * k + 0] = s0.x;
        w[4 * k + 1] = s0.y;
        w[4 * k + 2] = s1.x;
        w[4 * k + 3] = s1.y;
#else
        w[4 * k + 0] = __fadd_rn(w[4 * k + 0], __fmul_rn(q0.x, f));
        w[4 * k + 1] = __fadd_rn(w[4 * k + 1], __fmul_rn(q0.y, f));
        w[4 * k + 2] = __fadd_rn(w[4 * k + 2], __fmul_rn(q1.x, f));
        w[4 * k + 3] = __fadd_rn(w[4 * k + 3], __fmul_rn(q1.y, f));
#endif
    }
}

template <int B>
__global__ void __launch_bounds__(kReduceThreads) taco_shard_reduce_kernel(const ReduceArgs args)
{
    constexpr int LPB = B / kLaneCodes;   // lanes per block
    constexpr int kRec = B + 8;
    const int64_t total = args.nblocks * LPB;
    const int P = args.num_shards;
    grid_launch_dependents();
    grid_dependency_wait();   // the shards may come from the previous kernel

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         g - (threadIdx.x & 31) < total;  // whole warps iterate together
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool active = g < total;
        const int64_t k = active ? g / LPB : 0;
        const int part = static_cast<int>(g % LPB);
        const int64_t off = k * kRec;

        float w[kLaneCodes];
#pragma unroll
        for (int i = 0; i < kLaneCodes; i++)
            w[i] = 0.f;

        // W = sum_p q_p * (s_p / alpha_p) in shard order, the loads of up to
        // kBatch shards in flight at a time.  The shard loop is unrolled to
        // the maximum shard count so every shard pointer is a fixed kernel
        // parameter (no indexed parameter access).
#pragma unroll
        for (int p0 = 0; p0 < kMaxShards; p0 += kBatch) {
            if (p0 < P) {
                uint4 codes[kBatch];
                uint2 meta[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; i++) {
                    if (p0 + i < P && active) {
                        const uint8_t *rec = args.shards[p0 + i] + off;
                        codes[i] = ldg_codes16(rec + kLaneCodes * part);
                        meta[i] = ldg_nc_u2(rec + B);
                    } else {
                        codes[i] = make_uint4(0u, 0u, 0u, 0u);
                        meta[i] = make_uint2(0x3f800000u, 0u);  // alpha = 1, s = 0
                    }
                }
#pragma unroll
                for (int i = 0; i < kBatch; i++) {
                    if (p0 + i < P) {
                        // s_p / alpha_p (within 2 ulp; alpha_p <= 1e15 is far from
                        // the range where the fast quotient underflows).
                        const float f = __fdividef(__uint_as_float(meta[i].y), __uint_as_float(meta[i].x));
                        accumulate_shard(w, codes[i], f);
                    }
                }
            }
        }

        // Energy |W|^2 and max|W| over the block's lanes.
        float2 e2 = make_float2(0.f, 0.f);
        float wmax = 0.f;
#pragma unroll
        for (int i = 0; i < kLaneCodes; i += 2) {
            const float2 wi = make_float2(w[i], w[i + 1]);
            e2 = fma2(wi, wi, e2);
            wmax = max3(wmax, fabsf(w[i]), fabsf(w[i + 1]));
        }
        float e = e2.x + e2.y;
#pragma unroll
        for (int d = 1; d < LPB; d <<= 1) {
            e = e + __shfl_xor_sync(kFullMask, e, d);
            wmax = fmaxf(wmax, __shfl_xor_sync(kFullMask, wmax, d));
        }

        const float m = e * (1.0f / B);
        const float alpha = __fdiv_rn(kTau, __fsqrt_rn(m + kEps));
        float s = 0.f;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (wmax > 0.f) {
            s = __fdiv_rn(__fmul_rn(alpha, wmax), kQmax);
            const float kq = __fdiv_rn(kQmax, wmax);
            const float2 k2 = make_float2(kq, kq);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float2 u0 = mul2(make_float2(w[4 * j], w[4 * j + 1]), k2);
                const float2 u1 = mul2(make_float2(w[4 * j + 2], w[4 * j + 3]), k2);
                o[j] = e4m3x2_from_float2(u0.x, u0.y) | (e4m3x2_from_float2(u1.x, u1.y) << 16);
            }
            out = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (active) {
            uint8_t *rec = args.out + off;
            // Records are 8-byte aligned: two 8-byte stores per lane.
            *reinterpret_cast<uint2 *>(rec + kLaneCodes * part) = make_uint2(out.x, out.y);
            *reinterpret_cast<uint2 *>(rec + kLaneCodes * part + 8) = make_uint2(out.z, out.w);
            if (part == 0)
                *reinterpret_cast<uint2 *>(rec + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(s));
        }
    }
}

template <int B>
KernelInfo info()
{
    return KernelInfo{reinterpret_cast<void *>(&taco_shard_reduce_kernel<B>), 0, kReduceThreads, B / kLaneCodes,
                      kReduceThreads / 32};
}

}  // namespace

KernelInfo reduce_kernel_info(int block)
{
    switch (block) {
    case 64: return info<64>();
    case 128: return info<128>();
    case 256: return info<256>();
    default: return KernelInfo{};
    }
}

cudaError_t launch_reduce(int block, const ReduceArgs &args, int grid, cudaStream_t stream)
{
    const KernelInfo ki = reduce_kernel_info(block);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    ReduceArgs a = args;
    void *params[] = {&a};
    return launch_kernel(ki.fn, grid, ki.threads, 0, stream, params);
}

}  // namespace taco
