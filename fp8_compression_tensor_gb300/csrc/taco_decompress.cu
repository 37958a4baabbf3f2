// taco_decompress.cu -- the fused receiver-side kernel of TACO (Algorithm 1,
// lines 19-24; Eqs. 11-13; the paper's fused_ash_decompress_kernel) for GB300
// (sm_103a): one HBM pass, no intermediate writes.
//
// Work decomposition mirrors the compress kernel: each warp pipelines tiles
// of 32 consecutive records (16 for B = 256) through shared memory with bulk
// (TMA) copies on per-stage mbarriers.  A tile of records is contiguous, so
// one bulk copy fetches it; the record stride (B + 8 bytes) already keeps a
// lane's 8-byte reads free of bank conflicts.  Each lane decodes its block's
// codes two at a time (E4M3x2 -> F16x2 -> FP32, exact), runs the
// Walsh-Hadamard butterflies in registers on FP32x2 pairs, applies one
// per-block factor and converts to bf16 two at a time.  Output blocks are
// staged in padded shared-memory slots and leave by per-lane bulk stores.
//
// Arithmetic order.  (1/sqrt B) H_B (q s) / alpha = (H_B q) * (s / sqrt B / alpha)
// in real arithmetic; the kernel rotates the decoded codes (whose sums are
// exact in FP32 for all but extreme code mixes) and applies the factor
// c = (s * (1/sqrt B)) / alpha once, which differs from the literal order only
// by FP32 rounding.
#include "taco_device.cuh"
#include "taco_kernels.h"

namespace taco {
namespace {

template <int B>
struct DecompressShape {
    static constexpr int kLanesPerBlock = (B <= 128) ? 1 : 2;
    static constexpr int kTileBlocks = 32 / kLanesPerBlock;
    static constexpr int kLaneElems = B / kLanesPerBlock;
    static constexpr int kPairs = kLaneElems / 2;
    static constexpr int kRecBytes = B + 8;
    // Each lane stages its 2B/L output bytes in its own slot, padded by 16
    // bytes so that the lanes' 16-byte writes fall in distinct banks.
    static constexpr int kLaneOutBytes = 2 * B / kLanesPerBlock;
    static constexpr int kOutSlotBytes = kLaneOutBytes + 16;
    static constexpr int kInTileBytes = kTileBlocks * kRecBytes;
    static constexpr int kOutTileBytes = 32 * kOutSlotBytes;
};

template <int B, int STAGES, int NOUT>
struct DecompressWarpSmem {
    using S = DecompressShape<B>;
    alignas(16) uint8_t in[STAGES][S::kInTileBytes];
    alignas(16) uint8_t out[NOUT][S::kOutTileBytes];
    alignas(8) uint64_t bar[STAGES];
};

// Issues the bulk load of one tile's records (an even number of them; an odd
// last record of the tensor is read from global memory by its lane instead).
template <int B>
__device__ __forceinline__ void decompress_issue_tile(const uint8_t *__restrict__ packed, int64_t nblocks,
                                                      int64_t tile, uint32_t in_stage, uint32_t bar, int lane)
{
    using S = DecompressShape<B>;
    const int64_t blk0 = tile * S::kTileBlocks;
    const int nvalid = static_cast<int>(nblocks - blk0 < S::kTileBlocks ? nblocks - blk0 : S::kTileBlocks);
    const int neven = nvalid & ~1;
    if (lane == 0) {
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(neven) * S::kRecBytes);
        if (neven > 0)
            bulk_load(in_stage, packed + blk0 * S::kRecBytes, static_cast<uint32_t>(neven) * S::kRecBytes, bar);
    }
}

template <int N>
__device__ __forceinline__ void load_words(const uint8_t *src_gen, uint32_t src_smem, bool from_global,
                                           uint32_t (&w)[N])
{
#pragma unroll
    for (int j = 0; j < N / 2; j++) {
        uint2 v;
        if (from_global)
            v = *reinterpret_cast<const uint2 *>(src_gen + 8 * j);
        else
            v = lds64(src_smem + 8 * j);
        w[2 * j] = v.x;
        w[2 * j + 1] = v.y;
    }
}

template <int B, int STAGES, int NOUT, int WARPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB)
    taco_decompress_kernel(const uint8_t *__restrict__ packed, uint16_t *__restrict__ y, int64_t nblocks,
                      uint32_t *__restrict__ fault)
{
    using S = DecompressShape<B>;
    using Smem = DecompressWarpSmem<B, STAGES, NOUT>;
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
            decompress_issue_tile<B>(packed, nblocks, t, smem_addr(sm.in[s]), smem_addr(&sm.bar[s]), lane);
    }

    const int blk = lane / L;
    const int h = lane % L;
    const float rB = (B == 64) ? 0.125f : (B == 128) ? 0.0883883476483184405f : 0.0625f;

    int iter = 0;
    bool healthy = true;
    for (int64_t t = first; t < ntiles; t += stride, iter++) {
        const int stage = iter % STAGES;
        const uint32_t bar = smem_addr(&sm.bar[stage]);
        if (!mbar_wait_bounded(bar, (iter / STAGES) & 1, fault, kFaultDecompress)) {
            healthy = false;
            break;
        }
        const int64_t blk0 = t * S::kTileBlocks;
        const int nvalid = static_cast<int>(nblocks - blk0 < S::kTileBlocks ? nblocks - blk0 : S::kTileBlocks);
        const bool active = blk < nvalid;
        const bool from_global = (nvalid & 1) && blk == nvalid - 1;  // odd last record: not in the tile copy

        float2 v[NP];
        float factor = 0.f;
        if (active) {
            const uint8_t *rec_g = packed + (blk0 + blk) * S::kRecBytes;
            const uint32_t rec_s = smem_addr(sm.in[stage]) + blk * S::kRecBytes;
            uint2 meta;
            if (from_global)
                meta = *reinterpret_cast<const uint2 *>(rec_g + B);
            else
                meta = lds64(rec_s + B);
            const float alpha = __uint_as_float(meta.x);
            const float s = __uint_as_float(meta.y);
            factor = __fdiv_rn(__fmul_rn(s, rB), alpha);
            if constexpr (L == 1) {
                // Codes 4j..4j+3 sit in word j.  Pair i = (code 2i, code 2i+1)
                // after the butterfly on element bit 0.
                uint32_t w[B / 4];
                load_words<B / 4>(rec_g, rec_s, from_global, w);
#pragma unroll
                for (int j = 0; j < B / 4; j++) {
                    v[2 * j] = e4m3x2_butterfly(w[j] & 0xffffu);
                    v[2 * j + 1] = e4m3x2_butterfly(w[j] >> 16);
                }
            } else {
                // B = 256: half h forms c_j = q_j + (-1)^h q_{j+128} first.
                uint32_t wa[32], wb[32];
                load_words<32>(rec_g, rec_s, from_global, wa);
                load_words<32>(rec_g + 128, rec_s + 128, from_global, wb);
                const float sg = h ? -1.f : 1.f;
                const float2 sgn = make_float2(sg, sg);
#pragma unroll
                for (int j = 0; j < 32; j++) {
#pragma unroll
                    for (int half = 0; half < 2; half++) {
                        const uint32_t pa = half ? (wa[j] >> 16) : (wa[j] & 0xffffu);
                        const uint32_t pb = half ? (wb[j] >> 16) : (wb[j] & 0xffffu);
                        const float2 c = fma2(e4m3x2_to_float2(pb), sgn, e4m3x2_to_float2(pa));
                        v[2 * j + half] = make_float2(c.x + c.y, c.x - c.y);
                    }
                }
            }
            fwht_pairs<NP>(v);
        }

        // This stage's tile is consumed: refill it.
        fence_proxy_async_smem();
        __syncwarp();
        {
            const int64_t tn = t + STAGES * stride;
            if (tn < ntiles)
                decompress_issue_tile<B>(packed, nblocks, tn, smem_addr(sm.in[stage]), bar, lane);
        }

        // Scale, convert to bf16, stage and store.  Each lane's previous store
        // from this output buffer must have finished reading it.
        const int ob = iter % NOUT;
        bulk_wait_read<NOUT - 1>();
        if (active) {
            const float2 f2 = make_float2(factor, factor);
            const uint32_t slot = smem_addr(sm.out[ob]) + lane * S::kOutSlotBytes;
#pragma unroll
            for (int c = 0; c < NP / 4; c++) {
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 2; k++) {
                    const float2 a = mul2(v[4 * c + 2 * k], f2);
                    const float2 b = mul2(v[4 * c + 2 * k + 1], f2);
                    o[2 * k] = float2_to_bf16x2(a.x, a.y);
                    o[2 * k + 1] = float2_to_bf16x2(b.x, b.y);
                }
                sts128(slot + 16 * c, make_uint4(o[0], o[1], o[2], o[3]));
            }
            fence_proxy_async_smem();
            // One bulk store per lane: its block, or its half of a B = 256 block.
            bulk_store(y + (blk0 + blk) * B + h * (B / L), slot, S::kLaneOutBytes);
            bulk_commit();
        }
    }

    if (!healthy) {
        for (int s = 0; s < STAGES; s++) {
            int64_t i = s + static_cast<int64_t>((iter + STAGES - 1 - s) / STAGES) * STAGES;
            while (i >= 0 && first + i * stride >= ntiles)
                i -= STAGES;
            if (i >= 0)
                mbar_wait_bounded(smem_addr(&sm.bar[s]), static_cast<uint32_t>(i / STAGES) & 1u, fault,
                                  kFaultDecompress);
        }
    }
    bulk_wait_all<0>();
}

template <int B, int STAGES, int NOUT, int WARPS, int MINB>
struct DecompressConfig {
    static constexpr int kWarps = WARPS;
    static constexpr size_t kSmem = sizeof(DecompressWarpSmem<B, STAGES, NOUT>) * WARPS;
    static constexpr int kTileBlocks = DecompressShape<B>::kTileBlocks;
    static void *fn() { return reinterpret_cast<void *>(&taco_decompress_kernel<B, STAGES, NOUT, WARPS, MINB>); }
};

#ifndef TACO_DECOMPRESS64_CFG
#define TACO_DECOMPRESS64_CFG 4120
#endif
#ifndef TACO_DECOMPRESS128_CFG
#define TACO_DECOMPRESS128_CFG 2120
#endif
#ifndef TACO_DECOMPRESS256_CFG
#define TACO_DECOMPRESS256_CFG 2110
#endif
// Launch shapes, as four digits: stages, output buffers, warps per CTA, and
// the minimum CTAs per SM given to __launch_bounds__ (0: none).
using Decompress64 = DecompressConfig<64, TACO_DECOMPRESS64_CFG / 1000, TACO_DECOMPRESS64_CFG / 100 % 10, TACO_DECOMPRESS64_CFG / 10 % 10, TACO_DECOMPRESS64_CFG % 10>;
using Decompress128 = DecompressConfig<128, TACO_DECOMPRESS128_CFG / 1000, TACO_DECOMPRESS128_CFG / 100 % 10, TACO_DECOMPRESS128_CFG / 10 % 10, TACO_DECOMPRESS128_CFG % 10>;
using Decompress256 = DecompressConfig<256, TACO_DECOMPRESS256_CFG / 1000, TACO_DECOMPRESS256_CFG / 100 % 10, TACO_DECOMPRESS256_CFG / 10 % 10, TACO_DECOMPRESS256_CFG % 10>;

template <class C>
KernelInfo info()
{
    return KernelInfo{C::fn(), C::kSmem, C::kWarps * 32, C::kTileBlocks, C::kWarps};
}

}  // namespace

KernelInfo decompress_kernel_info(int block)
{
    switch (block) {
    case 64: return info<Decompress64>();
    case 128: return info<Decompress128>();
    case 256: return info<Decompress256>();
    default: return KernelInfo{};
    }
}

cudaError_t launch_decompress(int block, const void *packed, void *y, int64_t nblocks, uint32_t *fault, int grid,
                              cudaStream_t stream)
{
    const KernelInfo ki = decompress_kernel_info(block);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    const uint8_t *pp = static_cast<const uint8_t *>(packed);
    uint16_t *yp = static_cast<uint16_t *>(y);
    void *args[] = {&pp, &yp, &nblocks, &fault};
    return cudaLaunchKernel(ki.fn, dim3(grid), dim3(ki.threads), args, ki.smem, stream);
}

}  // namespace taco
