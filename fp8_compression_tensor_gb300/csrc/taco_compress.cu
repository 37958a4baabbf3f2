// taco_compress.cu -- the fused sender-side kernel of TACO (Algorithm 1, lines
// 4-16; Eqs. 5-10) for GB300 (sm_103a): one HBM pass per tensor.
//
// Work decomposition.  Each warp is an independent pipeline over "tiles" of
// 32 consecutive blocks (16 for B = 256).  For B <= 128 one lane owns one
// whole block; for B = 256 a lane pair owns a block.  Tiles are staged in
// shared memory by bulk (TMA) copies that complete on a per-stage mbarrier,
// STAGES tiles ahead of the one being computed.  A lane reads its block from
// its own padded slot (padding keeps the 16-byte reads free of bank
// conflicts), keeps it in registers, and computes everything there:
//   energy (Eq. 6)   sum of squares with packed FP32x2 FMAs,
//   rotation (Eq. 8) in-register Walsh-Hadamard butterflies on FP32x2 pairs,
//   scales (Eqs. 7, 9) and the E4M3 conversion (Eq. 10), two codes per cvt.
// Records are written to a shared-memory staging buffer in the packed layout
// (Section 4.4.2) and leave with one bulk store per tile.
//
// Arithmetic order.  The rotation is applied to the unscaled block: with
// y = H_B G, Z = alpha y / sqrt(B) and Z / s = Q_max y / max|y| in real
// arithmetic, so the kernel takes u = y * (Q_max / max|y|) and
// s = alpha * max|y| * (1/sqrt B) / Q_max.  This differs from the literal
// order only by FP32 rounding.
#include "taco_device.cuh"
#include "taco_kernels.h"

#ifndef TACO_COMPRESS_MIXED_UNPACK
#define TACO_COMPRESS_MIXED_UNPACK 1
#endif

namespace taco {
namespace {

template <int B>
struct CompressShape {
    static constexpr int kLanesPerBlock = (B <= 128) ? 1 : 2;
    static constexpr int kTileBlocks = 32 / kLanesPerBlock;        // blocks per warp tile
    static constexpr int kLaneElems = B / kLanesPerBlock;          // elements a lane owns
    static constexpr int kPairs = kLaneElems / 2;                  // FP32x2 registers a lane owns
    static constexpr int kSlotBytes = 2 * B + 16;                  // padded input slot per block
    static constexpr int kRecBytes = B + 8;                        // packed record
    static constexpr int kInTileBytes = kTileBlocks * kSlotBytes;
    static constexpr int kOutTileBytes = kTileBlocks * kRecBytes;  // multiple of 16
};

template <int B, int STAGES, int NOUT>
struct CompressWarpSmem {
    using S = CompressShape<B>;
    alignas(16) uint8_t in[STAGES][S::kInTileBytes];
    alignas(16) uint8_t out[NOUT][S::kOutTileBytes];
    alignas(8) uint64_t bar[STAGES];
};

// Issues the bulk loads of one tile into stage `stage` (every lane calls it).
template <int B>
__device__ __forceinline__ void compress_issue_tile(const uint16_t *__restrict__ x, int64_t nblocks, int64_t tile,
                                                    uint32_t in_stage, uint32_t bar, int lane)
{
    using S = CompressShape<B>;
    const int64_t blk0 = tile * S::kTileBlocks;
    const int nvalid = static_cast<int>(nblocks - blk0 < S::kTileBlocks ? nblocks - blk0 : S::kTileBlocks);
    if (lane == 0)
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid) * 2u * B);
    __syncwarp();
    // Lane `lane` copies bytes [part*2B/L, (part+1)*2B/L) of block lane/L.
    const int blk = lane / S::kLanesPerBlock;
    const int part = lane % S::kLanesPerBlock;
    if (blk < nvalid) {
        constexpr uint32_t kPartBytes = 2u * B / S::kLanesPerBlock;
        const uint16_t *src = x + (blk0 + blk) * B + part * (B / S::kLanesPerBlock);
        bulk_load(in_stage + blk * S::kSlotBytes + part * kPartBytes, src, kPartBytes, bar);
    }
}

// Energy partial sums and FWHT of a lane's data for B <= 128: the lane holds
// the whole block.  v[i] ends as (y[2i], y[2i+1]).
template <int B>
__device__ __forceinline__ float compress_rotate_whole(uint32_t slot, float2 (&v)[B / 2])
{
    constexpr int NP = B / 2;
    float2 acc[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        acc[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < B / 8; c++) {
        const uint4 raw = lds128(slot + 16 * c);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = 4 * c + k;
#if TACO_COMPRESS_MIXED_UNPACK
            // Butterfly on element bit 0 straight from the bf16 pair; the
            // energy comes from its outputs: (a+b)^2 + (a-b)^2 = 2(a^2 + b^2).
            v[i] = bf16x2_butterfly(w[k]);
            acc[i % 8] = fma2(v[i], v[i], acc[i % 8]);
#else
            const float2 g = bf16x2_to_float2(w[k]);
            acc[i % 8] = fma2(g, g, acc[i % 8]);
            v[i] = make_float2(g.x + g.y, g.x - g.y);  // butterfly on element bit 0
#endif
        }
    }
    fwht_pairs<NP>(v);
    // Tree-sum the 16 partial sums.
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; i++)
            acc[i] = add2(acc[i], acc[i + w]);
#if TACO_COMPRESS_MIXED_UNPACK
    return (acc[0].x + acc[0].y) * 0.5f;
#else
    return acc[0].x + acc[0].y;
#endif
}

// Same for B = 256 with a lane pair per block: lane half h first forms
// c_j = G_j + (-1)^h G_{j+128} (the butterfly on element bit 7), then runs the
// remaining seven stages on its 128 values, which become y[128h .. 128h+127].
// Returns the sum of squares of the lane's own half of G.
__device__ __forceinline__ float compress_rotate_half256(uint32_t slot, int h, float2 (&v)[64])
{
    float2 acc[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        acc[i] = make_float2(0.f, 0.f);
    const float sg = h ? -1.f : 1.f;
    const float2 sgn = make_float2(sg, sg);
#pragma unroll
    for (int c = 0; c < 16; c++) {
        const uint4 ra = lds128(slot + 16 * c);        // elements 8c .. 8c+7
        const uint4 rb = lds128(slot + 256 + 16 * c);  // elements 128+8c .. 128+8c+7
        const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
        const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = 4 * c + k;
            const float2 a = bf16x2_to_float2(wa[k]);
            const float2 b = bf16x2_to_float2(wb[k]);
            const float2 own = h ? b : a;
            acc[i % 8] = fma2(own, own, acc[i % 8]);
            const float2 cc = fma2(b, sgn, a);          // a + b or a - b, one rounding
            v[i] = make_float2(cc.x + cc.y, cc.x - cc.y);
        }
    }
    fwht_pairs<64>(v);
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; i++)
            acc[i] = add2(acc[i], acc[i + w]);
    return acc[0].x + acc[0].y;
}

template <int NP>
__device__ __forceinline__ float abs_max(const float2 (&v)[NP])
{
    float m0 = 0.f, m1 = 0.f;
#pragma unroll
    for (int i = 0; i < NP; i += 2) {
        m0 = max3(m0, fabsf(v[i].x), fabsf(v[i].y));
        m1 = max3(m1, fabsf(v[i + 1].x), fabsf(v[i + 1].y));
    }
    return fmaxf(m0, m1);
}

// Encodes a lane's NP pairs to E4M3 (u = y * k) into NP/2 words.
template <int NP>
__device__ __forceinline__ void encode_pairs(const float2 (&v)[NP], float k, uint32_t (&cw)[NP / 2])
{
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int i = 0; i < NP; i += 2) {
        const float2 u0 = mul2(v[i], k2);
        const float2 u1 = mul2(v[i + 1], k2);
        cw[i / 2] = e4m3x2_from_float2(u0.x, u0.y) | (e4m3x2_from_float2(u1.x, u1.y) << 16);
    }
}

template <int B, int STAGES, int NOUT, int WARPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB)
    taco_compress_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ packed, int64_t nblocks,
                    uint32_t *__restrict__ fault)
{
    using S = CompressShape<B>;
    using Smem = CompressWarpSmem<B, STAGES, NOUT>;
    constexpr int L = S::kLanesPerBlock;
    constexpr int NP = S::kPairs;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Smem &sm = reinterpret_cast<Smem *>(smem_raw)[warp];

    const int64_t ntiles = (nblocks + S::kTileBlocks - 1) / S::kTileBlocks;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * WARPS;
    if (first >= ntiles)
        return;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; s++)
            mbar_init(smem_addr(&sm.bar[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();

#pragma unroll
    for (int s = 0; s < STAGES; s++) {
        const int64_t t = first + s * stride;
        if (t < ntiles)
            compress_issue_tile<B>(x, nblocks, t, smem_addr(sm.in[s]), smem_addr(&sm.bar[s]), lane);
    }

    const int blk = lane / L;   // block of the tile this lane works on
    const int h = lane % L;     // which half (B = 256)
    const float rB = (B == 64) ? 0.125f : (B == 128) ? 0.0883883476483184405f : 0.0625f;

    int iter = 0;
    bool healthy = true;
    for (int64_t t = first; t < ntiles; t += stride, iter++) {
        const int stage = iter % STAGES;
        const uint32_t bar = smem_addr(&sm.bar[stage]);
        if (!mbar_wait_bounded(bar, (iter / STAGES) & 1, fault, kFaultCompress)) {
            healthy = false;
            break;
        }
        const int64_t blk0 = t * S::kTileBlocks;
        const int nvalid = static_cast<int>(nblocks - blk0 < S::kTileBlocks ? nblocks - blk0 : S::kTileBlocks);
        const bool active = blk < nvalid;

        // Load the block into registers, rotate it, and take its energy.
        float2 v[NP];
        float sumsq = 0.f;
        const uint32_t slot = smem_addr(sm.in[stage]) + blk * S::kSlotBytes;
        if (active) {
            if constexpr (L == 1)
                sumsq = compress_rotate_whole<B>(slot, v);
            else
                sumsq = compress_rotate_half256(slot, h, v);
        }

        // The stage's slots are consumed: refill them with tile t + STAGES*stride.
        fence_proxy_async_smem();
        __syncwarp();
        {
            const int64_t tn = t + STAGES * stride;
            if (tn < ntiles)
                compress_issue_tile<B>(x, nblocks, tn, smem_addr(sm.in[stage]), bar, lane);
        }

        // Scales (Eqs. 6, 7, 9) and codes (Eq. 10).
        float ymax = active ? abs_max<NP>(v) : 0.f;
        if constexpr (L == 2) {
            sumsq = sumsq + __shfl_xor_sync(kFullMask, sumsq, 1);
            ymax = fmaxf(ymax, __shfl_xor_sync(kFullMask, ymax, 1));
        }
        const float m = sumsq * (1.0f / B);
        const float sigma = __fsqrt_rn(m + kEps);
        const float alpha = __fdiv_rn(kTau, sigma);
        float s = 0.f, k = 0.f;
        if (ymax > 0.f) {
            s = __fdiv_rn(__fmul_rn(__fmul_rn(alpha, ymax), rB), kQmax);
            k = __fdiv_rn(kQmax, ymax);
        }
        uint32_t cw[NP / 2];
        if (ymax > 0.f) {
            encode_pairs<NP>(v, k, cw);
        } else {
#pragma unroll
            for (int i = 0; i < NP / 2; i++)
                cw[i] = 0u;
        }

        // Stage the record in shared memory (the previous store from this
        // buffer must have finished reading it).
        const int ob = iter % NOUT;
        if (lane == 0)
            bulk_wait_read<NOUT - 1>();
        __syncwarp();
        const uint32_t rec = smem_addr(sm.out[ob]) + blk * S::kRecBytes;
        if (active) {
            if constexpr (L == 1) {
#pragma unroll
                for (int j = 0; j < NP / 4; j++)
                    sts64(rec + 8 * j, cw[2 * j], cw[2 * j + 1]);
            } else {
                // Half h writes codes [128h, 128h+128); the second half of the
                // pair writes its chunks in a rotated order (chunk j+8 at step
                // j) so that the two halves hit different banks.
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int jr = (j + 8) & 15;
                    const uint32_t a = h ? cw[2 * jr] : cw[2 * j];
                    const uint32_t b = h ? cw[2 * jr + 1] : cw[2 * j + 1];
                    sts64(rec + (h ? 128 + 8 * jr : 8 * j), a, b);
                }
            }
            if (h == 0)
                sts64(rec + B, __float_as_uint(alpha), __float_as_uint(s));
        }
        fence_proxy_async_smem();
        __syncwarp();

        // Write the tile's records: one bulk store for an even count; an odd
        // last record goes out with plain stores.
        const int neven = nvalid & ~1;
        if (lane == 0 && neven > 0) {
            bulk_store(packed + blk0 * S::kRecBytes, smem_addr(sm.out[ob]), neven * S::kRecBytes);
            bulk_commit();
        }
        if ((nvalid & 1) && blk == nvalid - 1) {
            uint8_t *dst = packed + (blk0 + blk) * S::kRecBytes;
            const uint8_t *src = sm.out[ob] + blk * S::kRecBytes;
            for (int o = h * 8; o < S::kRecBytes; o += 8 * L)
                *reinterpret_cast<uint2 *>(dst + o) = *reinterpret_cast<const uint2 *>(src + o);
        }
    }

    if (!healthy) {
        // Let copies still in flight land before the CTA's shared memory is
        // released: for each stage, wait (bounded) for the last tile issued
        // into it.  Tile i of this warp went to stage i % STAGES as phase
        // i / STAGES; tiles i < iter + STAGES were issued.
        for (int s = 0; s < STAGES; s++) {
            int64_t i = s + static_cast<int64_t>((iter + STAGES - 1 - s) / STAGES) * STAGES;
            while (i >= 0 && first + i * stride >= ntiles)
                i -= STAGES;
            if (i >= 0)
                mbar_wait_bounded(smem_addr(&sm.bar[s]), static_cast<uint32_t>(i / STAGES) & 1u, fault,
                                  kFaultCompress);
        }
    }
    if (lane == 0)
        bulk_wait_all<0>();
}

template <int B, int STAGES, int NOUT, int WARPS, int MINB>
struct CompressConfig {
    static constexpr int kWarps = WARPS;
    static constexpr size_t kSmem = sizeof(CompressWarpSmem<B, STAGES, NOUT>) * WARPS;
    static constexpr int kTileBlocks = CompressShape<B>::kTileBlocks;
    static void *fn() { return reinterpret_cast<void *>(&taco_compress_kernel<B, STAGES, NOUT, WARPS, MINB>); }
};

#ifndef TACO_COMPRESS64_CFG
#define TACO_COMPRESS64_CFG 3110
#endif
#ifndef TACO_COMPRESS128_CFG
#define TACO_COMPRESS128_CFG 2110
#endif
#ifndef TACO_COMPRESS256_CFG
#define TACO_COMPRESS256_CFG 2110
#endif
// Launch shapes, as four digits: stages, output buffers, warps per CTA, and
// the minimum CTAs per SM given to __launch_bounds__ (0: none).
using Compress64 = CompressConfig<64, TACO_COMPRESS64_CFG / 1000, TACO_COMPRESS64_CFG / 100 % 10, TACO_COMPRESS64_CFG / 10 % 10, TACO_COMPRESS64_CFG % 10>;
using Compress128 = CompressConfig<128, TACO_COMPRESS128_CFG / 1000, TACO_COMPRESS128_CFG / 100 % 10, TACO_COMPRESS128_CFG / 10 % 10, TACO_COMPRESS128_CFG % 10>;
using Compress256 = CompressConfig<256, TACO_COMPRESS256_CFG / 1000, TACO_COMPRESS256_CFG / 100 % 10, TACO_COMPRESS256_CFG / 10 % 10, TACO_COMPRESS256_CFG % 10>;

template <class C>
KernelInfo info()
{
    return KernelInfo{C::fn(), C::kSmem, C::kWarps * 32, C::kTileBlocks, C::kWarps};
}

}  // namespace

KernelInfo compress_kernel_info(int block)
{
    switch (block) {
    case 64: return info<Compress64>();
    case 128: return info<Compress128>();
    case 256: return info<Compress256>();
    default: return KernelInfo{};
    }
}

cudaError_t launch_compress(int block, const void *x, void *packed, int64_t nblocks, uint32_t *fault, int grid,
                            cudaStream_t stream)
{
    const KernelInfo ki = compress_kernel_info(block);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    uint8_t *pp = static_cast<uint8_t *>(packed);
    void *args[] = {&xp, &pp, &nblocks, &fault};
    return cudaLaunchKernel(ki.fn, dim3(grid), dim3(ki.threads), args, ki.smem, stream);
}

}  // namespace taco
