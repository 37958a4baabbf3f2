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
// Layout.  B/8 consecutive lanes share a block; each lane owns 8 elements,
// i.e. 8 bytes of codes per shard, read with coalesced 8-byte loads (a warp
// reads whole records).  Energy and maximum are reduced across the block's
// lanes with xor-shuffles (every lane ends with the same bits).
#include "taco_device.cuh"
#include "taco_kernels.h"

namespace taco {
namespace {

constexpr int kReduceThreads = 256;

__device__ __forceinline__ uint2 ldg_nc_u2(const uint8_t *p)
{
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

template <int B>
__global__ void __launch_bounds__(kReduceThreads) taco_shard_reduce_kernel(const ReduceArgs args)
{
    constexpr int LPB = B / 8;            // lanes per block
    constexpr int kRec = B + 8;
    const int64_t total = args.nblocks * LPB;
    const int P = args.num_shards;

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         g - (threadIdx.x & 31) < total;  // whole warps iterate together
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool active = g < total;
        const int64_t k = active ? g / LPB : 0;
        const int part = static_cast<int>(g % LPB);
        const int64_t off = k * kRec;

        float2 w[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
            w[i] = make_float2(0.f, 0.f);

        // W = sum_p q_p * (s_p / alpha_p) in shard order, four shards' loads in flight at a time.
        for (int p0 = 0; p0 < P; p0 += 4) {
            uint2 codes[4], meta[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                if (p0 + i < P && active) {
                    const uint8_t *rec = args.shards[p0 + i] + off;
                    codes[i] = ldg_nc_u2(rec + 8 * part);
                    meta[i] = ldg_nc_u2(rec + B);
                } else {
                    codes[i] = make_uint2(0u, 0u);
                    meta[i] = make_uint2(0x3f800000u, 0u);  // alpha = 1, s = 0
                }
            }
#pragma unroll
            for (int i = 0; i < 4; i++) {
                if (p0 + i < P) {
                    const float f = __fdiv_rn(__uint_as_float(meta[i].y), __uint_as_float(meta[i].x));
                    // Each product rounded on its own, then added: a shard and
                    // its negation cancel exactly, as in an FP32 sum of decoded
                    // shards.
                    w[0] = add_rounded_product(w[0], e4m3x2_to_float2(codes[i].x & 0xffffu), f);
                    w[1] = add_rounded_product(w[1], e4m3x2_to_float2(codes[i].x >> 16), f);
                    w[2] = add_rounded_product(w[2], e4m3x2_to_float2(codes[i].y & 0xffffu), f);
                    w[3] = add_rounded_product(w[3], e4m3x2_to_float2(codes[i].y >> 16), f);
                }
            }
        }

        // Energy |W|^2 and max|W| over the block's lanes.
        float2 e2 = mul2(w[0], w[0]);
        e2 = fma2(w[1], w[1], e2);
        e2 = fma2(w[2], w[2], e2);
        e2 = fma2(w[3], w[3], e2);
        float e = e2.x + e2.y;
        float wmax = max3(fabsf(w[0].x), fabsf(w[0].y), fabsf(w[1].x));
        wmax = max3(wmax, fabsf(w[1].y), fabsf(w[2].x));
        wmax = max3(wmax, fabsf(w[2].y), fabsf(w[3].x));
        wmax = fmaxf(wmax, fabsf(w[3].y));
#pragma unroll
        for (int d = 1; d < LPB; d <<= 1) {
            e = e + __shfl_xor_sync(kFullMask, e, d);
            wmax = fmaxf(wmax, __shfl_xor_sync(kFullMask, wmax, d));
        }

        const float m = e * (1.0f / B);
        const float alpha = __fdiv_rn(kTau, __fsqrt_rn(m + kEps));
        float s = 0.f;
        uint32_t c0 = 0u, c1 = 0u;
        if (wmax > 0.f) {
            s = __fdiv_rn(__fmul_rn(alpha, wmax), kQmax);
            const float kq = __fdiv_rn(kQmax, wmax);
            const float2 k2 = make_float2(kq, kq);
            const float2 u0 = mul2(w[0], k2), u1 = mul2(w[1], k2);
            const float2 u2 = mul2(w[2], k2), u3 = mul2(w[3], k2);
            c0 = e4m3x2_from_float2(u0.x, u0.y) | (e4m3x2_from_float2(u1.x, u1.y) << 16);
            c1 = e4m3x2_from_float2(u2.x, u2.y) | (e4m3x2_from_float2(u3.x, u3.y) << 16);
        }
        if (active) {
            uint8_t *rec = args.out + off;
            *reinterpret_cast<uint2 *>(rec + 8 * part) = make_uint2(c0, c1);
            if (part == 0)
                *reinterpret_cast<uint2 *>(rec + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(s));
        }
    }
}

template <int B>
KernelInfo info()
{
    return KernelInfo{reinterpret_cast<void *>(&taco_shard_reduce_kernel<B>), 0, kReduceThreads, 0, kReduceThreads / 32};
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
    return cudaLaunchKernel(ki.fn, dim3(grid), dim3(ki.threads), params, 0, stream);
}

}  // namespace taco
