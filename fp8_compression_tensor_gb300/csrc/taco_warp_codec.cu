// taco_warp_codec.cu -- compress and decompress for B = 32, the smallest
// block of the paper's block-size ablation ("TACO: Efficient Communication
// Compression of Intermediate Tensors for Scalable Tensor-Parallel LLM
// Training", Section 5.3.3, Table 2), on the CUDA cores, for GB300 (sm_103a).
//
// One lane per block: the whole Walsh-Hadamard butterfly (a, b) -> (a + b,
// a - b) at strides 1..16, which gives H_32 y in Sylvester order, and the
// block's energy and maximum stay in registers (a 32-element block is too
// short for a tensor-core tile row of 128 bytes, and a warp per block would
// spend every per-block scalar on 32 elements only).  Every scheme of the
// tensor-core kernels is supported (variants and code formats; see
// taco_compress.cu), with the same arithmetic shortcuts: the rotation is
// applied to the unscaled block, the codes are Cvt(y Q_max / max|y|) and the
// decoder multiplies H q by one factor.
#include "taco_device.cuh"
#include "taco_kernels.h"

namespace taco {
namespace {

constexpr int kWarpThreads = 256;   // blocks per CTA and pass

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h)
{
    return __uint_as_float(h << 16);
}

// In-register Walsh-Hadamard transform of n values (strides 1 .. n/2).
template <int N>
__device__ __forceinline__ void fwht_regs(float (&v)[N])
{
#pragma unroll
    for (int h = 1; h < N; h <<= 1) {
#pragma unroll
        for (int i = 0; i < N; i++) {
            if ((i & h) == 0) {
                const float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
        }
    }
}

constexpr int kLaneBlock = 32;   // B of the lane-per-block kernels

__global__ void __launch_bounds__(kWarpThreads) taco_lane_compress_kernel(const uint16_t *__restrict__ x,
                                                                          uint8_t *__restrict__ packed,
                                                                          int64_t nblocks, const Scheme scheme)
{
    constexpr int B = kLaneBlock, kRec = B + 8;
    grid_launch_dependents();
    grid_dependency_wait();
    const bool rotate = scheme.variant != 2;
    const bool adaptive = scheme.variant == 0 || scheme.variant == 3;
    const bool dual_scale = scheme.variant != 3;
    const float rr = rotate ? 0.176776695296636881f : 1.0f;   // 1/sqrt(32) in binary32
    const float qmax = code_qmax(scheme.code);
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * kWarpThreads + threadIdx.x; k < nblocks;
         k += static_cast<int64_t>(gridDim.x) * kWarpThreads) {
        float v[B];
        const uint16_t *src = x + k * B;
#pragma unroll
        for (int q = 0; q < B / 8; q++) {   // blocks start at 64-byte multiples
            const uint4 w = *reinterpret_cast<const uint4 *>(src + 8 * q);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                v[8 * q + 2 * j] = bf16_bits_to_float(ws[j] & 0xffffu);
                v[8 * q + 2 * j + 1] = bf16_bits_to_float(ws[j] >> 16);
            }
        }
        float e = 0.f;
#pragma unroll
        for (int i = 0; i < B; i++)
            e = fmaf(v[i], v[i], e);
        if (rotate)
            fwht_regs<B>(v);
        float ymax = 0.f;
#pragma unroll
        for (int i = 0; i < B; i++)
            ymax = fmaxf(ymax, fabsf(v[i]));
        const float alpha = adaptive ? __fdiv_rn(kTau, __fsqrt_rn(e * (1.0f / B) + kEps)) : 1.0f;
        float s = 0.f, kq = 0.f;
        if (!dual_scale) {
            s = 1.0f;
            kq = __fmul_rn(alpha, rr);
        } else if (ymax > 0.f) {
            s = __fdiv_rn(__fmul_rn(__fmul_rn(alpha, ymax), rr), qmax);
            kq = __fdiv_rn(qmax, ymax);
        }
        uint32_t cw[B / 4];
#pragma unroll
        for (int j = 0; j < B / 4; j++)
            cw[j] = ymax > 0.f ? encode4(scheme.code, v[4 * j] * kq, v[4 * j + 1] * kq, v[4 * j + 2] * kq,
                                         v[4 * j + 3] * kq)
                               : 0u;
        uint8_t *rec = packed + k * kRec;   // 8-byte aligned
#pragma unroll
        for (int j = 0; j < B / 8; j++)
            *reinterpret_cast<uint2 *>(rec + 8 * j) = make_uint2(cw[2 * j], cw[2 * j + 1]);
        *reinterpret_cast<uint2 *>(rec + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(s));
    }
}

__global__ void __launch_bounds__(kWarpThreads) taco_lane_decompress_kernel(const uint8_t *__restrict__ packed,
                                                                            uint16_t *__restrict__ y,
                                                                            int64_t nblocks, const Scheme scheme)
{
    constexpr int B = kLaneBlock, kRec = B + 8;
    grid_launch_dependents();
    grid_dependency_wait();
    const bool rotate = scheme.variant != 2;
    const float rr = rotate ? 0.176776695296636881f : 1.0f;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * kWarpThreads + threadIdx.x; k < nblocks;
         k += static_cast<int64_t>(gridDim.x) * kWarpThreads) {
        const uint8_t *rec = packed + k * kRec;
        const uint2 meta = *reinterpret_cast<const uint2 *>(rec + B);
        const float f = __fdiv_rn(__fmul_rn(__uint_as_float(meta.y), rr), __uint_as_float(meta.x));
        float v[B];
#pragma unroll
        for (int j = 0; j < B / 8; j++) {
            const uint2 w = *reinterpret_cast<const uint2 *>(rec + 8 * j);
            const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
            for (int h = 0; h < 2; h++) {
                if (scheme.code == 2) {
                    float2 lo, hi;
                    int8x4_to_float(ws[h], lo, hi);
                    v[8 * j + 4 * h] = lo.x;
                    v[8 * j + 4 * h + 1] = lo.y;
                    v[8 * j + 4 * h + 2] = hi.x;
                    v[8 * j + 4 * h + 3] = hi.y;
                } else {
                    const float2 lo = scheme.code == 0 ? e4m3x2_to_float2(ws[h] & 0xffffu)
                                                       : e5m2x2_to_float2(ws[h] & 0xffffu);
                    const float2 hi = scheme.code == 0 ? e4m3x2_to_float2(ws[h] >> 16) : e5m2x2_to_float2(ws[h] >> 16);
                    v[8 * j + 4 * h] = lo.x;
                    v[8 * j + 4 * h + 1] = lo.y;
                    v[8 * j + 4 * h + 2] = hi.x;
                    v[8 * j + 4 * h + 3] = hi.y;
                }
            }
        }
        if (rotate)
            fwht_regs<B>(v);
        uint16_t *dst = y + k * B;
#pragma unroll
        for (int q = 0; q < B / 8; q++) {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                o[j] = float2_to_bf16x2(v[8 * q + 2 * j] * f, v[8 * q + 2 * j + 1] * f);
            *reinterpret_cast<uint4 *>(dst + 8 * q) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

KernelInfo lane_info(bool compress)
{
    void *fn = compress ? reinterpret_cast<void *>(&taco_lane_compress_kernel)
                        : reinterpret_cast<void *>(&taco_lane_decompress_kernel);
    return KernelInfo{fn, 0, kWarpThreads, kWarpThreads, kWarpThreads / 32};
}

}  // namespace

KernelInfo warp_codec_info(int block, bool compress)
{
    return block == 32 ? lane_info(compress) : KernelInfo{};
}

cudaError_t launch_warp_compress(int block, Scheme scheme, const void *x, void *packed, int64_t nblocks, int grid,
                                 cudaStream_t stream)
{
    const KernelInfo ki = warp_codec_info(block, true);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    uint8_t *pp = static_cast<uint8_t *>(packed);
    void *args[] = {&xp, &pp, &nblocks, &scheme};
    return launch_kernel(ki.fn, grid, ki.threads, 0, stream, args);
}

cudaError_t launch_warp_decompress(int block, Scheme scheme, const void *packed, void *y, int64_t nblocks, int grid,
                                   cudaStream_t stream)
{
    const KernelInfo ki = warp_codec_info(block, false);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    const uint8_t *pp = static_cast<const uint8_t *>(packed);
    uint16_t *yp = static_cast<uint16_t *>(y);
    void *args[] = {&pp, &yp, &nblocks, &scheme};
    return launch_kernel(ki.fn, grid, ki.threads, 0, stream, args);
}

}  // namespace taco
