// taco_warp_codec.cu -- compress and decompress for B = 32, the smallest
// block of the paper's block-size ablation ("TACO: Efficient Communication
// Compression of Intermediate Tensors for Scalable Tensor-Parallel LLM
// Training", Section 5.3.3, Table 2), on the CUDA cores, for GB300 (sm_103a).
//
// One lane per block: the whole Walsh-Hadamard butterfly (a, b) -> (a + b,
// a - b) at strides 1..16, which gives H_32 y in Sylvester order, and the
// block's energy and maximum stay in registers (a 32-element block is too
// short for a tensor-core tile row of 128 bytes, and a warp per block would
// spend every per-block scalar on 32 elements only).  A warp moves its 32
// consecutive blocks (2 KB of bf16, 1280 bytes of records) with fully
// coalesced 16-byte accesses through a swizzled shared-memory staging buffer,
// so each warp-wide load or store touches four or five 128-byte lines instead
// of sixteen to thirty-two.  Every scheme of the tensor-core kernels is
// supported (variants and code formats; see taco_compress.cu), with the same
// arithmetic shortcuts: the rotation is applied to the unscaled block, the
// codes are Cvt(y Q_max / max|y|) and the decoder multiplies H q by one factor.
#include "taco_device.cuh"
#include "taco_kernels.h"

namespace taco {
namespace {

constexpr int kWarpThreads = 256;   // threads of a CTA; a warp codes 32 consecutive blocks per pass
constexpr int kLaneBlock = 32;      // B of the lane-per-block kernels
constexpr int kRec32 = kLaneBlock + 8;
constexpr int kInUnits = 32 * kLaneBlock * 2 / 16;   // 16-byte units of a warp's 32 bf16 blocks (128)
constexpr int kRecUnits = 32 * kRec32 / 16;           // 16-byte units of its 32 records (80)

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h)
{
    return __uint_as_float(h << 16);
}

// Packed FP32x2 subtract (one issue for two IEEE subtractions).
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// In-register Walsh-Hadamard transform of n values (strides 1 .. n/2).
// Stride 1 pairs the two halves of a value pair and runs scalar; strides 2 ..
// n/2 butterfly neighbouring pairs with packed FP32x2 adds and subtracts (the
// same IEEE results per element, half the issue slots).
template <int N>
__device__ __forceinline__ void fwht_regs(float (&v)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = a + b;
        v[i + 1] = a - b;
    }
#pragma unroll
    for (int h = 2; h < N; h <<= 1) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            if ((i & h) == 0) {
                const float2 p = make_float2(v[i], v[i + 1]), q = make_float2(v[i + h], v[i + h + 1]);
                const float2 s = add2(p, q), d = sub2(p, q);
                v[i] = s.x;
                v[i + 1] = s.y;
                v[i + h] = d.x;
                v[i + h + 1] = d.y;
            }
        }
    }
}

// Slot of 16-byte unit c (elements 8(c % 4) .. 8(c % 4) + 7 of the warp's
// block c / 4) in the warp's staging buffer.  The XOR of the unit's low three
// bits with the next three spreads both access patterns over all eight
// 16-byte bank groups: the coalesced copy (lane l moves units l + 32j) and the
// per-block access (lane i moves units 4i + q) each take four wavefronts per
// 512 bytes, the minimum.
__device__ __forceinline__ int unit_slot(int c)
{
    return (c & ~7) | ((c ^ (c >> 3)) & 7);
}

// Asynchronous 16-byte copy global -> shared (both 16-byte aligned), tracked by
// this thread's copy groups; the bytes are visible to the thread after
// cp_async_wait and to its warp after a __syncwarp() that follows it.
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// At most N of this thread's most recent copy groups may still be in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp's 32 input blocks at k0 (2 KB) into its staging buffer, one copy
// group per lane (empty when the group of blocks is not complete).
__device__ __forceinline__ void stage_blocks_async(uint4 *buf, const uint16_t *x, int64_t k0, int64_t nblocks,
                                                   int lane)
{
    if (k0 + 32 <= nblocks) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + k0 * kLaneBlock);
#pragma unroll
        for (int j = 0; j < 4; j++)
            cp_async16(buf + unit_slot(lane + 32 * j), src + lane + 32 * j);
    }
    cp_async_commit();
}

// A warp's 32 records at k0 (1280 bytes) into its staging buffer, likewise.
__device__ __forceinline__ void stage_records_async(uint4 *buf, const uint8_t *packed, int64_t k0, int64_t nblocks,
                                                    int lane)
{
    if (k0 + 32 <= nblocks) {
        const uint4 *src = reinterpret_cast<const uint4 *>(packed + k0 * kRec32);
        cp_async16(buf + lane, src + lane);
        cp_async16(buf + lane + 32, src + lane + 32);
        if (lane < kRecUnits - 64)
            cp_async16(buf + lane + 64, src + lane + 64);
    }
    cp_async_commit();
}

#ifndef TACO_LANE_IN_BUFS
#define TACO_LANE_IN_BUFS 3
#endif
// Compress: input staging buffers per warp, a ring with the next two groups'
// copies in flight (two buffers: 78.9 us, three: 76.9 us on 16384 x 8192).
constexpr int kInBufs = TACO_LANE_IN_BUFS;

// INT8: the rotating schemes with INT8 codes (scalar products before the
// integer rounding, see encode4_scaled) are their own instantiation, so the
// FP8 kernel carries no format branch around its packed products.
template <bool INT8>
__global__ void __launch_bounds__(kWarpThreads) taco_lane_compress_kernel(const uint16_t *__restrict__ x,
                                                                          uint8_t *__restrict__ packed,
                                                                          int64_t nblocks, const Scheme scheme)
{
    constexpr int B = kLaneBlock, kRec = kRec32;
    // Per warp: a ring of kInBufs buffers of 32 input blocks (2 KB each; the
    // next groups are copied in while this one is coded) and its 32 records
    // (1280 B).
    __shared__ __align__(16) uint4 stage_in[kWarpThreads / 32][kInBufs][kInUnits];
    __shared__ __align__(16) uint4 stage_rec[kWarpThreads / 32][kRecUnits];
    grid_launch_dependents();
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 *srec = stage_rec[warp];
    uint8_t *srec_b = reinterpret_cast<uint8_t *>(srec);
    const bool rotate = scheme.variant != 2;
    const bool adaptive = scheme.variant == 0 || scheme.variant == 3;
    const bool dual_scale = scheme.variant != 3;
    const float rr = rotate ? 0.176776695296636881f : 1.0f;   // 1/sqrt(32) in binary32
    const float qmax = code_qmax(scheme.code);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpThreads;
    int64_t k0 = (static_cast<int64_t>(blockIdx.x) * (kWarpThreads / 32) + warp) * 32;
#pragma unroll
    for (int j = 0; j < kInBufs - 1; j++)
        stage_blocks_async(stage_in[warp][j], x, k0 + j * stride, nblocks, lane);
    for (int buf = 0; k0 < nblocks; k0 += stride, buf = buf + 1 == kInBufs ? 0 : buf + 1) {
        // Coalesced: the warp's 32 blocks are 2 KB of contiguous input; the
        // next groups' copies are in flight while this one is coded.
        stage_blocks_async(stage_in[warp][buf == 0 ? kInBufs - 1 : buf - 1], x, k0 + (kInBufs - 1) * stride,
                           nblocks, lane);
        const int64_t k = k0 + lane;              // this lane's block
        const bool full = k0 + 32 <= nblocks;     // warp-uniform
        if (!full && k >= nblocks)
            continue;
        float v[B];
        if (full) {
            const uint4 *sin = stage_in[warp][buf];
            cp_async_wait<kInBufs - 1>();         // this group's copies (all but the newest)
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint4 u = sin[unit_slot(4 * lane + q)];
                const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    v[8 * q + 2 * j] = bf16_bits_to_float(ws[j] & 0xffffu);
                    v[8 * q + 2 * j + 1] = bf16_bits_to_float(ws[j] >> 16);
                }
            }
            __syncwarp();                         // read before the buffer's next copy is issued
        } else {
            // The tensor's last, partial group of 32 blocks: one lane per block.
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
        }
        float2 e2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < B; i += 2) {
            const float2 vi = make_float2(v[i], v[i + 1]);
            e2[(i >> 1) & 1] = fma2(vi, vi, e2[(i >> 1) & 1]);
        }
        const float2 e01 = add2(e2[0], e2[1]);
        const float e = e01.x + e01.y;
        if (rotate)
            fwht_regs<B>(v);
        float ymax = 0.f;
#pragma unroll
        for (int i = 0; i < B; i += 2)
            ymax = max3(ymax, fabsf(v[i]), fabsf(v[i + 1]));
        const float alpha = adaptive ? __fdiv_rn(kTau, __fsqrt_rn(e * (1.0f / B) + kEps)) : 1.0f;
        // A tiny rotation (max|y| < 2^-100) is scaled by 2^64 before its codes
        // are formed, so that Q_max / max|y| cannot overflow.
        const bool tiny = dual_scale && rotate && ymax > 0.f && ymax < kTinyValue;
        const float pre = tiny ? kTinyUp : 1.0f;
        float s = 0.f, kq = 0.f;
        if (!dual_scale) {
            s = 1.0f;
            kq = __fmul_rn(alpha, rr);
        } else if (ymax > 0.f) {
            s = __fdiv_rn(__fmul_rn(__fmul_rn(alpha, ymax), rr), qmax);
            kq = __fdiv_rn(qmax, __fmul_rn(ymax, pre));
        }
        if (tiny) {
#pragma unroll
            for (int i = 0; i < B; i++)
                v[i] = __fmul_rn(v[i], kTinyUp);
        }
        uint32_t cw[B / 4];
        const float2 k2 = make_float2(kq, kq);
        if ((rotate || !dual_scale) && INT8) {
            // INT8: scalar products before the integer rounding (encode4_scaled).
#pragma unroll
            for (int j = 0; j < B / 4; j++)
                cw[j] = ymax > 0.f ? encode4_scaled(2, make_float2(v[4 * j], v[4 * j + 1]),
                                                    make_float2(v[4 * j + 2], v[4 * j + 3]), kq)
                                   : 0u;
        } else if (rotate || !dual_scale) {
#pragma unroll
            for (int j = 0; j < B / 4; j++) {
                const float2 u0 = mul2(make_float2(v[4 * j], v[4 * j + 1]), k2);
                const float2 u1 = mul2(make_float2(v[4 * j + 2], v[4 * j + 3]), k2);
                cw[j] = ymax > 0.f ? encode4(scheme.code, u0.x, u0.y, u1.x, u1.y) : 0u;
            }
        } else if (s >= kDivFastMin) {
            // DS only: G / s correctly rounded, as Eq. (10) writes it (bf16
            // ratios often land exactly on rounding midpoints).
            const float srcp = __frcp_rn(s);
#pragma unroll
            for (int j = 0; j < B / 4; j++) {
                const float2 u0 = div2_by(make_float2(v[4 * j], v[4 * j + 1]), s, srcp);
                const float2 u1 = div2_by(make_float2(v[4 * j + 2], v[4 * j + 3]), s, srcp);
                cw[j] = encode4(scheme.code, u0.x, u0.y, u1.x, u1.y);
            }
        } else {
            // DS only with a tiny (or zero) s: IEEE division.
#pragma unroll
            for (int j = 0; j < B / 4; j++) {
                float u[4];
#pragma unroll
                for (int h = 0; h < 4; h++)
                    u[h] = s > 0.f ? __fdiv_rn(v[4 * j + h], s) : 0.f;
                cw[j] = ymax > 0.f ? encode4(scheme.code, u[0], u[1], u[2], u[3]) : 0u;
            }
        }
        if (full) {
            // The warp's 32 records are 1280 contiguous bytes: stage, then store coalesced.
            __syncwarp();                         // the previous pass has read the buffer
            uint8_t *r = srec_b + lane * kRec;    // 8-byte aligned; two wavefronts per store
#pragma unroll
            for (int j = 0; j < B / 8; j++)
                *reinterpret_cast<uint2 *>(r + 8 * j) = make_uint2(cw[2 * j], cw[2 * j + 1]);
            *reinterpret_cast<uint2 *>(r + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(s));
            __syncwarp();
            uint4 *dst = reinterpret_cast<uint4 *>(packed + k0 * kRec);   // 1280-byte multiple offset
            dst[lane] = srec[lane];
            dst[lane + 32] = srec[lane + 32];
            if (lane < kRecUnits - 64)
                dst[lane + 64] = srec[lane + 64];
        } else {
            uint8_t *rec = packed + k * kRec;   // 8-byte aligned
#pragma unroll
            for (int j = 0; j < B / 8; j++)
                *reinterpret_cast<uint2 *>(rec + 8 * j) = make_uint2(cw[2 * j], cw[2 * j + 1]);
            *reinterpret_cast<uint2 *>(rec + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(s));
        }
    }
    cp_async_wait<0>();   // no copy may land in shared memory after the CTA is gone
}

__global__ void __launch_bounds__(kWarpThreads) taco_lane_decompress_kernel(const uint8_t *__restrict__ packed,
                                                                            uint16_t *__restrict__ y,
                                                                            int64_t nblocks, const Scheme scheme)
{
    constexpr int B = kLaneBlock, kRec = kRec32;
    // Per warp: two buffers of 32 records (the next group is copied in while
    // this one is decoded) and its 32 output blocks (2 KB).
    __shared__ __align__(16) uint4 stage_out[kWarpThreads / 32][kInUnits];
    __shared__ __align__(16) uint4 stage_rec[kWarpThreads / 32][2][kRecUnits];
    grid_launch_dependents();
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 *sout = stage_out[warp];
    const bool rotate = scheme.variant != 2;
    const float rr = rotate ? 0.176776695296636881f : 1.0f;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpThreads;
    int64_t k0 = (static_cast<int64_t>(blockIdx.x) * (kWarpThreads / 32) + warp) * 32;
    stage_records_async(stage_rec[warp][0], packed, k0, nblocks, lane);
    for (int buf = 0; k0 < nblocks; k0 += stride, buf ^= 1) {
        // Coalesced: the warp's 32 records are 1280 contiguous bytes; the next
        // group's copy is in flight while this one is decoded.
        stage_records_async(stage_rec[warp][buf ^ 1], packed, k0 + stride, nblocks, lane);
        const int64_t k = k0 + lane;
        const bool full = k0 + 32 <= nblocks;     // warp-uniform
        if (!full && k >= nblocks)
            continue;
        const uint8_t *rec;
        if (full) {
            cp_async_wait<1>();                   // this group's copies (all but the newest)
            __syncwarp();
            rec = reinterpret_cast<const uint8_t *>(stage_rec[warp][buf]) + lane * kRec;
        } else {
            rec = packed + k * kRec;
        }
        const uint2 meta = *reinterpret_cast<const uint2 *>(rec + B);
        const float sv = __uint_as_float(meta.y), av = __uint_as_float(meta.x);
        float f = __fdiv_rn(__fmul_rn(sv, rr), av);
        // A tiny factor (below 2^-100, or flushed to zero by the division) is
        // formed 2^64 times larger and the products are scaled back after it.
        const bool tiny = sv > 0.f && f < kTinyValue;
        if (tiny)
            f = __fdiv_rn(__fmul_rn(__fmul_rn(sv, kTinyUp), rr), av);
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
        if (full)
            __syncwarp();                         // read before the buffer's next copy is issued
        if (rotate)
            fwht_regs<B>(v);
        uint4 o[B / 8];
#pragma unroll
        for (int q = 0; q < B / 8; q++) {
            uint32_t t[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float2 g = mul2(make_float2(v[8 * q + 2 * j], v[8 * q + 2 * j + 1]), make_float2(f, f));
                if (tiny)
                    g = make_float2(__fmul_rn(g.x, kTinyDown), __fmul_rn(g.y, kTinyDown));
                t[j] = float2_to_bf16x2(g.x, g.y);
            }
            o[q] = make_uint4(t[0], t[1], t[2], t[3]);
        }
        if (full) {
            // The warp's 32 output blocks are 2 KB contiguous: stage, then store coalesced.
            __syncwarp();                         // the previous pass has read the buffer
#pragma unroll
            for (int q = 0; q < B / 8; q++)
                sout[unit_slot(4 * lane + q)] = o[q];
            __syncwarp();
            uint4 *dst = reinterpret_cast<uint4 *>(y + k0 * B);
#pragma unroll
            for (int j = 0; j < 4; j++)
                dst[lane + 32 * j] = sout[unit_slot(lane + 32 * j)];
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(y + k * B);
#pragma unroll
            for (int q = 0; q < B / 8; q++)
                dst[q] = o[q];
        }
    }
    cp_async_wait<0>();   // no copy may land in shared memory after the CTA is gone
}

KernelInfo lane_info(bool compress, int code)
{
    void *fn = !compress ? reinterpret_cast<void *>(&taco_lane_decompress_kernel)
               : code == 2 ? reinterpret_cast<void *>(&taco_lane_compress_kernel<true>)
                           : reinterpret_cast<void *>(&taco_lane_compress_kernel<false>);
    return KernelInfo{fn, 0, kWarpThreads, kWarpThreads, kWarpThreads / 32};
}

}  // namespace

KernelInfo warp_codec_info(int block, bool compress, int code)
{
    return block == 32 ? lane_info(compress, code) : KernelInfo{};
}

cudaError_t launch_warp_compress(int block, Scheme scheme, const void *x, void *packed, int64_t nblocks, int grid,
                                 cudaStream_t stream)
{
    const KernelInfo ki = warp_codec_info(block, true, scheme.code);
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
    const KernelInfo ki = warp_codec_info(block, false, scheme.code);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    const uint8_t *pp = static_cast<const uint8_t *>(packed);
    uint16_t *yp = static_cast<uint16_t *>(y);
    void *args[] = {&pp, &yp, &nblocks, &scheme};
    return launch_kernel(ki.fn, grid, ki.threads, 0, stream, args);
}

}  // namespace taco
