// taco_decompress.cu -- TACO's fused receiver-side kernel (Algorithm 1, its
// decompression loop; Eqs. 11-13; the paper's fused_ash_decompress_kernel) with the
// inverse rotation on the tensor cores (tcgen05), for GB300 (sm_103a).
//
// For a tile of blocks, the E4M3 codes of each block form one row of A and
// Y = A H^T (H symmetric) gives H q for every block at once: the codes are
// the MMA's 8-bit operand (.kind::f8f6f4), H holds +-1 in E4M3, products are
// exact and accumulate in FP32 in tensor memory.  G' = Y * (s / sqrt(B) / alpha)
// per block is Eqs. (11)-(13) up to FP32 summation order.  Near zero the
// factor would be subnormal: below 2^-100 it is formed 2^64 times larger and
// the products are scaled back by 2^-64.
//
// Scheduling: one CTA per tile, one CTA per SM resident (shared memory); a
// running CTA takes its own tile, then the tiles of CTAs it cancels before
// they start (cluster launch control, taco_sched.cuh).
//
// Roles in a CTA:
//   warp 0    bulk-copies each tile of records (contiguous, B + 8 bytes each)
//             into a ring of raw stages;
//   warp 1    allocates tensor memory and issues the MMAs of a tile into one
//             of two to four accumulators (tile i into accumulator i mod
//             their number; M = 128 rows, N = 128, K = 32 per MMA);
//   warps 2-5 "transposers": each thread takes one MMA row, copies its codes
//             from the record into the 128-byte swizzled K-major A layout,
//             and writes the block's factor s / sqrt(B) / alpha;
//   warps 6.. epilogue, EPG groups of 4 warps taking rotating tiles: each
//             thread reads its row of the accumulator from
//             TMEM, scales it by the factor, converts two values per cvt to
//             bf16 into a swizzled output tile, which one thread writes with
//             2-D TMA stores (rows past the tensor's end are not written).
// Block sizes: 128 (one block per row, H_128), 64 (two blocks per row,
// H = diag(H_64, H_64)), 256 and 512 (two or four rows of 128 codes per
// block, H_128 on each and a butterfly across the parts' neighbouring TMEM
// lanes for the H_2 or H_4 factor of H_B).
//
// Ablations (Scheme): E5M2 codes are the MMA's operand as E5M2 (H in E5M2);
// INT8 codes (A16: the 8-bit integer MMA kind does not exist on sm_103a) go
// through .kind::f16: a code v becomes the f16 1152 + v exactly (the bytes
// v ^ 0x80 under the exponent byte 0x64 give 1024 + (v + 128)), H holds +-1 in
// f16, and since H 1 = B e_0 the epilogue subtracts 1152 B from each block's
// first column (1152 from every column without rotation); all sums are
// integers below 2^24, so the decoded H v is exact.  DS only puts the
// identity in place of H; the factor is s / sqrt(B) / alpha, or s / alpha
// without rotation.
#include <cstring>

#include <cuda.h>

#include "taco_device.cuh"
#include "taco_kernels.h"
#include "taco_sched.cuh"
#include "taco_tcgen05.cuh"

namespace taco {
namespace {

constexpr int kDRows = 128;        // MMA rows per tile
// Threads: loader, MMA, 4 transposer warps and EPG groups of 4 epilogue warps.
__host__ __device__ constexpr int dthreads(int epg) { return 192 + 128 * epg; }
constexpr int kGroup = 128;        // threads of the transposer / epilogue groups

template <int B, int RS, int AS, int NOUT, int A16, int EPG>
struct TcDecompressLayout {
    // B = 256 and 512: each block is B / 128 A rows of 128 codes (its parts),
    // in neighbouring rows of the tile.
    static constexpr bool kSplit = B > 128;
    static constexpr int kBlocksPerRow = B == 64 ? 2 : 1;
    static constexpr int kRowsPerBlock = kSplit ? B / 128 : 1;
    static constexpr int kTileBlocks = kDRows * kBlocksPerRow / kRowsPerBlock;
    static constexpr int kPartCodes = kSplit ? 128 : B;            // codes of one block (part) in a row
    static constexpr int kRowCodes = kPartCodes * kBlocksPerRow;   // 128 or 256
    static constexpr int kElem = A16 ? 2 : 1;                      // bytes per code in the A operand
    static constexpr int kAChunks = kRowCodes * kElem / 128;       // 128-byte chunks of an A row
    static constexpr int kAccCols = 128;                           // TMEM columns per tile
    static constexpr int kRec = B + 8;
    static constexpr int kRawBytes = kTileBlocks * kRec;
    static constexpr int kAStageBytes = kDRows * kRowCodes * kElem;
    static constexpr int kAChunkBytes = kDRows * 128;
    static constexpr int kHChunkBytes = 128 * 128;                 // 128 rows of H, 128 bytes of K
    static constexpr int kHBytes = kAChunks * kHChunkBytes;        // K chunks of H = those of an A row
    static constexpr int kOutRows = kSplit ? kDRows : kTileBlocks; // rows of the y view per tile
    static constexpr int kOutChunks = B == 64 ? 1 : kPartCodes / 64;   // 64-element chunks of a y row
    static constexpr int kOutChunkBytes = kOutRows * 128;
    static constexpr int kOutBytes = kOutChunks * kOutChunkBytes;
    // Accumulators in tensor memory (512 columns): up to four, so that more
    // than two epilogue groups can hold one each while the MMA fills the next.
    static constexpr int kNumAcc = 4 * kAccCols <= 512 ? 4 : 2;
    // Factor slots: the transposer writes item i's factors after the MMA of
    // item i - AS, which needed item i - AS - kNumAcc's accumulator back from
    // the epilogue (which had read that item's factors): AS + kNumAcc slots
    // are never overwritten before they are read.
    static constexpr int FS = AS + kNumAcc;
    static_assert(NOUT % EPG == 0, "every epilogue group owns NOUT / EPG output tiles");
    // Offsets from the 1024-byte aligned base.
    static constexpr int kOffA = 0;
    static constexpr int kOffH = kOffA + AS * kAStageBytes;
    static constexpr int kOffOut = kOffH + kHBytes;
    static constexpr int kOffRaw = kOffOut + NOUT * kOutBytes;
    static constexpr int kOffFac = kOffRaw + RS * kRawBytes;      // 16-byte aligned (kRawBytes % 16 == 0)
    // Tile scheduler.  The loader publishes item i after the raw-stage
    // barrier of item i - RS, when the epilogue has read items up to
    // i - RS - AS - 2: a published-tile slot is reused only after every
    // reader is done with it.
    static_assert(kTileRing >= RS + AS + kNumAcc + EPG, "published-tile slot reused too early");
    static constexpr int kOffSched = kOffFac + FS * kTileBlocks * 4;   // 16-byte aligned
    static_assert(kOffSched % 16 == 0, "cancel responses need 16-byte alignment");
    static constexpr int kOffBar = kOffSched + kSchedBytes;
    static constexpr int kNumBars = 2 * RS + 2 * AS + 2 * kNumAcc + 2 * NOUT + FS;
    static constexpr int kOffTmem = kOffBar + 8 * kNumBars;
    static constexpr int kBytes = kOffTmem + 16;
    static constexpr int kSmem = kBytes + 1024;
    static constexpr int kTmemCols = kNumAcc * kAccCols;
};

// The MMA's B operand, K-major, 128-byte swizzle, in E4M3 (+1 = 0x38,
// -1 = 0xB8) or E5M2 (+1 = 0x3C, -1 = 0xBC): H_128 for B = 128 / 256,
// diag(H_64, H_64) for B = 64, the identity when `rotate` is false.  Written
// by the threads of warps 1 and up, before their dependency wait: warp 0's
// thread 0 issues the first loads right after that wait and would otherwise
// hold the CTA's set-up barrier for its share.
template <int B>
__device__ void write_hadamard_f8_sw128(uint8_t *h, bool e5m2, bool rotate)
{
    const uint32_t plus = e5m2 ? 0x3Cu : 0x38u, minus = e5m2 ? 0xBCu : 0xB8u;
    if (threadIdx.x < 32)
        return;
    for (int idx = threadIdx.x - 32; idx < 128 * 8; idx += blockDim.x - 32) {
        const int n = idx / 8, u = idx % 8;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t word = 0;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const int k = 16 * u + 4 * q + b;
                uint32_t code;
                if (!rotate)
                    code = (n == k) ? plus : 0x00u;
                else if (B == 64)
                    code = (n / 64 != k / 64) ? 0x00u : ((__popc((n & 63) & (k & 63)) & 1) ? minus : plus);
                else
                    code = (__popc(n & k) & 1) ? minus : plus;
                word |= code << (8 * b);
            }
            w[q] = word;
        }
        *reinterpret_cast<uint4 *>(h + n * 128 + ((u ^ (n & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The same in f16 (+1 = 0x3C00, -1 = 0xBC00): two 128-byte K chunks of 64
// columns each, written by the same threads.
template <int B>
__device__ void write_hadamard_f16_sw128(uint8_t *h, bool rotate)
{
    if (threadIdx.x < 32)
        return;
    for (int idx = threadIdx.x - 32; idx < 128 * 16; idx += blockDim.x - 32) {
        const int n = idx / 16, ua = idx % 16;   // row, 16-byte unit along K (8 columns)
        const int c = ua / 8, u = ua % 8;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int k = 8 * ua + 2 * q + e;
                uint32_t v;
                if (!rotate)
                    v = (n == k) ? 0x3C00u : 0u;
                else if (B == 64)
                    v = (n / 64 != k / 64) ? 0u : ((__popc((n & 63) & (k & 63)) & 1) ? 0xBC00u : 0x3C00u);
                else
                    v = (__popc(n & k) & 1) ? 0xBC00u : 0x3C00u;
                word |= v << (16 * e);
            }
            w[q] = word;
        }
        *reinterpret_cast<uint4 *>(h + c * 16384 + n * 128 + ((u ^ (n & 7)) * 16)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int B, int RS, int AS, int NOUT, int A16, int EPG>
__global__ void __launch_bounds__(dthreads(EPG), 1)
    taco_decompress_kernel(const __grid_constant__ CUtensorMap tmap_y, const uint8_t *__restrict__ packed,
                              int64_t nblocks, uint32_t *__restrict__ fault, const Scheme scheme)
{
    using Lay = TcDecompressLayout<B, RS, AS, NOUT, A16, EPG>;
    constexpr int FS = Lay::FS;
    constexpr int NBG = NOUT / EPG;   // output tiles per epilogue group
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(base);
    const uint32_t bar0 = sbase + Lay::kOffBar;
    auto raw_full = [&](int s) { return bar0 + 8u * s; };
    auto raw_empty = [&](int s) { return bar0 + 8u * (RS + s); };
    auto a_full = [&](int j) { return bar0 + 8u * (2 * RS + j); };
    auto a_empty = [&](int j) { return bar0 + 8u * (2 * RS + AS + j); };
    constexpr int NACC = Lay::kNumAcc;
    auto acc_full = [&](int a) { return bar0 + 8u * (2 * RS + 2 * AS + a); };
    auto acc_empty = [&](int a) { return bar0 + 8u * (2 * RS + 2 * AS + NACC + a); };
    auto out_free = [&](int b) { return bar0 + 8u * (2 * RS + 2 * AS + 2 * NACC + b); };
    auto out_done = [&](int b) { return bar0 + 8u * (2 * RS + 2 * AS + 2 * NACC + NOUT + b); };
    auto fac_full = [&](int f) { return bar0 + 8u * (2 * RS + 2 * AS + 2 * NACC + 2 * NOUT + f); };
    const TileSched sched{sbase + Lay::kOffSched, fault, kFaultDecompress};
    float *factors = reinterpret_cast<float *>(base + Lay::kOffFac);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + Lay::kOffTmem);

    grid_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; s++) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), kGroup / 32);
        }
        for (int j = 0; j < AS; j++) {
            mbar_init(a_full(j), kGroup / 32);
            mbar_init(a_empty(j), 1);
        }
        for (int a = 0; a < NACC; a++) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), kGroup / 32);
        }
        for (int b = 0; b < NOUT; b++) {
            mbar_init(out_free(b), 1);
            mbar_init(out_done(b), kGroup / 32);
        }
        for (int f = 0; f < FS; f++)
            mbar_init(fac_full(f), kGroup / 32);
        sched.init();
        fence_mbar_init();
        prefetch_tmap(&tmap_y);
    }
    // The loader (thread 0) sends the first kSchedAhead tile requests and
    // starts its own tile's record copy (item 0) before the rest of the set-up.
    auto issue_tile = [&](int i, int64_t t) {
        const int s = i % RS;
        const int64_t blk0 = t * Lay::kTileBlocks;
        const int nvalid = static_cast<int>(nblocks - blk0 < Lay::kTileBlocks ? nblocks - blk0 : Lay::kTileBlocks);
        const uint32_t bytes = static_cast<uint32_t>(nvalid & ~1) * Lay::kRec;   // multiple of 16
        mbar_arrive_expect_tx(raw_full(s), bytes);
        if (bytes > 0)
            bulk_load(sbase + Lay::kOffRaw + s * Lay::kRawBytes, packed + blk0 * Lay::kRec, bytes, raw_full(s));
    };
    if (threadIdx.x == 0) {
        for (int j = 1; j <= kSchedAhead; j++)
            sched.request(j);
        // While the previous kernel drains: the records of its own tile and,
        // as a guess at the next rounds' tiles, one and more SM counts further on.
        for (int k = 0; k < kL2PrefetchDecompress; k++) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(k) * num_sms();
            if (t < gridDim.x) {
                const int64_t blk0 = t * Lay::kTileBlocks;
                const int64_t nv = nblocks - blk0 < Lay::kTileBlocks ? nblocks - blk0 : Lay::kTileBlocks;
                const uint32_t bytes = static_cast<uint32_t>(nv & ~1) * Lay::kRec;   // multiple of 16
                if (bytes > 0)
                    bulk_prefetch_l2(packed + blk0 * Lay::kRec, bytes);
            }
        }
        grid_dependency_wait();   // the input may come from the previous kernel
        sched.publish(0, blockIdx.x);
        issue_tile(0, blockIdx.x);
    }
    if (warp == 1)
        tmem_alloc(smem_addr(tmem_slot), Lay::kTmemCols);
    const bool rotate = scheme.variant != 2;   // DS only: no rotation
    const bool e5m2 = !A16 && scheme.code == 1;
    if constexpr (A16)
        write_hadamard_f16_sw128<B>(base + Lay::kOffH, rotate);
    else
        write_hadamard_f8_sw128<B>(base + Lay::kOffH, e5m2, rotate);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    grid_dependency_wait();   // before any global access of this thread
    cta_barrier();   // lanes of warps 0 and 1 took different paths above
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---- record loader ----------------------------------------------
        if (lane == 0) {
            int i = 1;                           // items 0 .. i-1 have been loaded
            int requested = kSchedAhead;         // requests 1 .. requested issued
            for (;; i++) {
                const int64_t t = sched.response(i);
                if (t < 0) {
                    sched.publish_end(i, EPG);
                    break;
                }
                sched.request(++requested);      // no failure seen yet: keep kSchedAhead in flight
                const int s = i % RS;
                if (i >= RS && !mbar_wait_bounded_thread(raw_empty(s), ((i / RS) - 1) & 1, fault, kFaultDecompress)) {
                    sched.publish_end(i, EPG);
                    break;
                }
                sched.publish(i, t);
                issue_tile(i, t);
            }
            // Responses still in flight and copies this thread issued must
            // land before the CTA can exit.
            sched.drain(i, requested);
            const int issued = i;
            for (int j = issued - RS > 0 ? issued - RS : 0; j < issued; j++)
                mbar_wait_bounded_thread(raw_full(j % RS), (j / RS) & 1, fault, kFaultDecompress);
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----------------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = A16    ? mma_idesc_f16_f32(kDRows, 128)
                                   : e5m2 ? mma_idesc_e5m2_f32(kDRows, 128)
                                          : mma_idesc_e4m3_f32(kDRows, 128);
            const uint32_t h0 = sbase + Lay::kOffH;
            int i = 0;
            for (;; i++) {
                if (sched.tile_thread(i) < 0)
                    break;
                const int j = i % AS, acc = i % NACC;
                if (i >= NACC &&
                    !mbar_wait_bounded_thread(acc_empty(acc), ((i / NACC) - 1) & 1, fault, kFaultDecompress))
                    break;
                if (!mbar_wait_bounded_thread(a_full(j), (i / AS) & 1, fault, kFaultDecompress))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * Lay::kAccCols);
                const uint32_t a_st = sbase + Lay::kOffA + j * Lay::kAStageBytes;
#pragma unroll
                for (int c = 0; c < Lay::kAChunks; c++) {
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {   // 32 bytes of K per MMA
                        const uint64_t ad = sw128_kmajor_desc(a_st + c * Lay::kAChunkBytes + 32 * kk);
                        const uint64_t bd = sw128_kmajor_desc(h0 + c * Lay::kHChunkBytes + 32 * kk);
                        const uint32_t accumulate = (c == 0 && kk == 0) ? 0u : 1u;
                        if constexpr (A16)
                            tc_mma_bf16(d, ad, bd, idesc, accumulate);
                        else
                            tc_mma_f8(d, ad, bd, idesc, accumulate);
                    }
                }
                tc_commit(a_empty(j));
                tc_commit(acc_full(acc));
            }
            if (i > 0)
                mbar_wait_bounded_thread(acc_full((i - 1) % NACC), ((i - 1) / NACC) & 1, fault, kFaultDecompress);
        }
    } else if (warp < 6) {
        // ---- transposers (warps 2..5): one MMA row per thread ---------------
        const int m = threadIdx.x - 64;    // 0..127
        const float rB = (B == 64)    ? 0.125f
                         : (B == 128) ? 0.0883883476483184405f
                         : (B == 256) ? 0.0625f
                                      : 0.0441941738241592203f;   // 1/sqrt(B) in binary32
        const float rr = rotate ? rB : 1.0f;
        for (int i = 0;; i++) {
            const int64_t t = sched.tile_warp(i);
            if (t < 0)
                break;
            const int s = i % RS, j = i % AS, fs = i % FS;
            if (!mbar_wait_bounded(raw_full(s), (i / RS) & 1, fault, kFaultDecompress))
                break;
            if (i >= AS && !mbar_wait_bounded(a_empty(j), ((i / AS) - 1) & 1, fault, kFaultDecompress))
                break;
            const int64_t blk0 = t * Lay::kTileBlocks;
            const int nvalid = static_cast<int>(nblocks - blk0 < Lay::kTileBlocks ? nblocks - blk0 : Lay::kTileBlocks);
            const uint32_t raw = sbase + Lay::kOffRaw + s * Lay::kRawBytes;
            const uint32_t a_row = sbase + Lay::kOffA + j * Lay::kAStageBytes + m * 128;
#pragma unroll
            for (int b = 0; b < Lay::kBlocksPerRow; b++) {
                constexpr int PC = Lay::kPartCodes;
                const int bl = (m * Lay::kBlocksPerRow + b) / Lay::kRowsPerBlock;   // block within the tile
                const int part = m % Lay::kRowsPerBlock;                             // B = 256 / 512: part
                // B = 512: the four parts of a record lie 128 bytes apart, on
                // the same banks, so part p reads its 8-byte pieces starting at
                // piece 4p (register pair q holds piece (q + 4p) mod 16) and
                // stores unit u at (u + 2p) mod 8: two wavefronts per read.
                constexpr bool kRot = Lay::kRowsPerBlock == 4;
                const int rot = kRot ? part : 0;
                uint32_t w[PC / 4];
                float f = 0.f;
                if (bl < nvalid) {
                    const bool from_global = (nvalid & 1) && bl == nvalid - 1;   // not in the bulk copy
                    const uint8_t *rg = packed + (blk0 + bl) * Lay::kRec;
                    const uint32_t rs = raw + bl * Lay::kRec;
#pragma unroll
                    for (int q = 0; q < PC / 8; q++) {
                        const int o = part * PC + 8 * ((q + 4 * rot) % (PC / 8));
                        const uint2 v = from_global ? *reinterpret_cast<const uint2 *>(rg + o) : lds64(rs + o);
                        w[2 * q] = v.x;
                        w[2 * q + 1] = v.y;
                    }
                    const uint2 meta = from_global ? *reinterpret_cast<const uint2 *>(rg + B) : lds64(rs + B);
                    const float sv = __uint_as_float(meta.y), av = __uint_as_float(meta.x);
                    f = __fdiv_rn(__fmul_rn(sv, rr), av);
                    // A tiny factor (below 2^-100, or flushed to zero by the
                    // division) is stored 2^64 times larger and negated: the
                    // epilogue then scales its products back by 2^-64.
                    if (sv > 0.f && f < kTinyValue)
                        f = -__fdiv_rn(__fmul_rn(__fmul_rn(sv, kTinyUp), rr), av);
                } else {
#pragma unroll
                    for (int q = 0; q < PC / 4; q++)
                        w[q] = 0u;
                }
                if (part == 0)
                    factors[fs * Lay::kTileBlocks + bl] = f;
                // Codes to the swizzled A row: 16 codes per 16-byte unit (8 in f16).
#pragma unroll
                for (int u = 0; u < PC / 16; u++) {
                    const int ur = (u + 2 * rot) % (PC / 16);     // the unit register group u holds
                    if constexpr (!A16) {
                        const int ua = b * (PC / 16) + ur;        // unit index along the A row
                        const int chunk = ua / 8, uc = ua % 8;
                        sts128(a_row + chunk * Lay::kAChunkBytes + ((uc ^ (m & 7)) * 16),
                               make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]));
                    } else {
                        // INT8 v -> f16 1152 + v: bytes (v ^ 0x80) under 0x64.
                        uint32_t hv[8];
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const uint32_t xb = w[4 * u + q] ^ 0x80808080u;
                            hv[2 * q] = __byte_perm(xb, 0x64646464u, 0x4140);
                            hv[2 * q + 1] = __byte_perm(xb, 0x64646464u, 0x4342);
                        }
#pragma unroll
                        for (int hh = 0; hh < 2; hh++) {
                            const int ua = 2 * (b * (PC / 16) + ur) + hh;
                            const int chunk = ua / 8, uc = ua % 8;
                            sts128(a_row + chunk * Lay::kAChunkBytes + ((uc ^ (m & 7)) * 16),
                                   make_uint4(hv[4 * hh], hv[4 * hh + 1], hv[4 * hh + 2], hv[4 * hh + 3]));
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(raw_empty(s));
                mbar_arrive(a_full(j));
                mbar_arrive(fac_full(fs));
            }
        }
    } else {
        // ---- epilogue (warps 6.., EPG groups of 4): one MMA row per thread ---
        // Group g takes the tiles i with i % EPG == g.
        const int grp = (warp - 6) / 4;
        const int et = threadIdx.x - 192 - kGroup * grp;   // 0..127 within the group
        const int q = warp & 3;
        const int m = 32 * q + lane;               // accumulator row
        for (int kt = 0;; kt++) {                  // kt: tiles this group has handled
            const int i = EPG * kt + grp;
            const int64_t t = sched.tile_warp(i);
            if (t < 0)
                break;
            const int acc = i % NACC, fs = i % FS, ob = grp * NBG + kt % NBG;
            if (!mbar_wait_bounded(acc_full(acc), (i / NACC) & 1, fault, kFaultDecompress))
                break;
            if (!mbar_wait_bounded(fac_full(fs), (i / FS) & 1, fault, kFaultDecompress))
                break;
            tc_fence_after_sync();
            float fb[Lay::kBlocksPerRow];
#pragma unroll
            for (int b = 0; b < Lay::kBlocksPerRow; b++)
                fb[b] = factors[fs * Lay::kTileBlocks + (m * Lay::kBlocksPerRow + b) / Lay::kRowsPerBlock];
            if (kt >= NBG) {
                if (et == 0) {
                    bulk_wait_read<NBG - 1>();
                    mbar_arrive(out_free(ob));
                }
                if (!mbar_wait_bounded(out_free(ob), ((kt / NBG) - 1) & 1, fault, kFaultDecompress))
                    break;
            }
            const uint32_t out = sbase + Lay::kOffOut + ob * Lay::kOutBytes;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(acc * Lay::kAccCols);
#pragma unroll
            for (int c = 0; c < Lay::kAccCols / 32; c++) {
                uint32_t r[32];
                tmem_ld32(taddr + 32 * c, r);
                tmem_ld_wait();
                const int e0 = 32 * c;                     // first element (column) of the chunk
                const int b = (B == 64) ? e0 / 64 : 0;     // block within the row (B = 64)
                if constexpr (A16) {                       // remove the f16 bias 1152 of the codes
                    constexpr int kBiasCols = Lay::kPartCodes;   // the length H was applied over
                    if (!rotate) {
#pragma unroll
                        for (int h = 0; h < 32; h++)
                            r[h] = __float_as_uint(__uint_as_float(r[h]) - 1152.0f);
                    } else if (e0 % kBiasCols == 0) {
                        r[0] = __float_as_uint(__uint_as_float(r[0]) - 1152.0f * kBiasCols);
                    }
                }
                if constexpr (Lay::kSplit) {   // H_B = H_2 / H_4 (x) H_128: finish across the parts' lanes
                    if (rotate) {   // lower lane a + b, upper lane a - b, as one fma each
                        const float sgn1 = (m & 1) ? -1.0f : 1.0f, sgn2 = (m & 2) ? -1.0f : 1.0f;
#pragma unroll
                        for (int h = 0; h < 32; h++) {
                            float v = __uint_as_float(r[h]);
                            v = fmaf(sgn1, v, __shfl_xor_sync(kFullMask, v, 1));
                            if constexpr (Lay::kRowsPerBlock == 4)
                                v = fmaf(sgn2, v, __shfl_xor_sync(kFullMask, v, 2));
                            r[h] = __float_as_uint(v);
                        }
                    }
                }
                // A negative factor is a tiny block's factor times -2^64: its
                // products are scaled back by 2^-64 (the rare pass below).
                float f = fb[b];
                if (__any_sync(kFullMask, f < 0.f)) {      // warp-uniform, rare
                    if (f < 0.f) {                         // the products, scaled back; then a factor 1
#pragma unroll
                        for (int h = 0; h < 32; h++)
                            r[h] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[h]), -f), kTinyDown));
                        f = 1.0f;
                    }
                }
                const float2 f2 = make_float2(f, f);
                const int row = (B == 64) ? 2 * m + b : m; // y row within the tile
                const int el = (B == 64) ? e0 % 64 : e0;   // element within the block row
#pragma unroll
                for (int uu = 0; uu < 4; uu++) {           // four 8-element units
                    uint32_t o[4];
#pragma unroll
                    for (int h = 0; h < 4; h++) {
                        const float2 v = mul2(make_float2(__uint_as_float(r[8 * uu + 2 * h]),
                                                          __uint_as_float(r[8 * uu + 2 * h + 1])), f2);
                        o[h] = float2_to_bf16x2(v.x, v.y);
                    }
                    const int e = el + 8 * uu;
                    const int oc = e / 64, u = (e % 64) / 8;
                    sts128(out + oc * Lay::kOutChunkBytes + row * 128 + ((u ^ (row & 7)) * 16),
                           make_uint4(o[0], o[1], o[2], o[3]));
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acc_empty(acc));
            fence_proxy_async_smem();
            __syncwarp();                               // one arrival per warp covers its lanes' writes
            if (lane == 0)
                mbar_arrive(out_done(ob));
            if (warp == 6 + 4 * grp) {   // the group's first warp stores the tile
                if (!mbar_wait_bounded(out_done(ob), (kt / NBG) & 1, fault, kFaultDecompress))
                    break;
                if (lane == 0) {
                    const int32_t y0 = static_cast<int32_t>(t * Lay::kOutRows);
#pragma unroll
                    for (int oc = 0; oc < Lay::kOutChunks; oc++)
                        tma_store_2d(&tmap_y, 64 * oc, y0, out + oc * Lay::kOutChunkBytes);
                    bulk_commit();
                }
            }
        }
        // The shared-memory sources of this thread's stores must be read
        // before the CTA exits; the writes themselves complete before the
        // grid does.
        if (et == 0)
            bulk_wait_read<0>();
    }

    tc_fence_before_sync();
    cta_barrier();   // every role ran lane-divergent code
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Lay::kTmemCols);
    }
}

template <int B, int RS, int AS, int NOUT, int A16, int EPG = 1>
struct TcDecompressConfig {
    using Lay = TcDecompressLayout<B, RS, AS, NOUT, A16, EPG>;
    static_assert(Lay::kSmem <= 227 * 1024, "shared memory budget");
    static_assert(Lay::kRawBytes % 16 == 0, "raw stage alignment");
    static void *fn() { return reinterpret_cast<void *>(&taco_decompress_kernel<B, RS, AS, NOUT, A16, EPG>); }
    static KernelInfo info()
    {
        return KernelInfo{fn(), static_cast<size_t>(Lay::kSmem), dthreads(EPG), Lay::kTileBlocks, 0};
    }
};

#ifndef TACO_DTC64_CFG
#define TACO_DTC64_CFG 422
#endif
#ifndef TACO_DTC128_CFG
#define TACO_DTC128_CFG 622
#endif
#ifndef TACO_DTC256_CFG
#define TACO_DTC256_CFG 323
#endif
#ifndef TACO_DTC512_CFG
#define TACO_DTC512_CFG 323
#endif
// Per block size, three digits: raw stages, A stages, output tiles.
#ifndef TACO_DEPG64
#define TACO_DEPG64 2
#endif
#ifndef TACO_DEPG128
#define TACO_DEPG128 2
#endif
#ifndef TACO_DEPG256
#define TACO_DEPG256 3
#endif
#ifndef TACO_DEPG512
#define TACO_DEPG512 3
#endif
// EPG: epilogue groups (3 for B = 256 and 512, whose epilogues carry the
// butterfly across the parts' lanes; 2 for B = 64 and 128, where two tiles'
// epilogues in flight shorten each launch's tail).
using DecompressTc64 =
    TcDecompressConfig<64, TACO_DTC64_CFG / 100, TACO_DTC64_CFG / 10 % 10, TACO_DTC64_CFG % 10, 0, TACO_DEPG64>;
using DecompressTc128 =
    TcDecompressConfig<128, TACO_DTC128_CFG / 100, TACO_DTC128_CFG / 10 % 10, TACO_DTC128_CFG % 10, 0, TACO_DEPG128>;
using DecompressTc256 =
    TcDecompressConfig<256, TACO_DTC256_CFG / 100, TACO_DTC256_CFG / 10 % 10, TACO_DTC256_CFG % 10, 0, TACO_DEPG256>;
using DecompressTc512 =
    TcDecompressConfig<512, TACO_DTC512_CFG / 100, TACO_DTC512_CFG / 10 % 10, TACO_DTC512_CFG % 10, 0, TACO_DEPG512>;
// INT8 codes (f16 operands: A stages and H twice as large).  B = 128, four
// digits: raw stages, A stages, output tiles, epilogue groups.
#ifndef TACO_DI8_128_CFG
#define TACO_DI8_128_CFG 3222
#endif
using DecompressI8x64 = TcDecompressConfig<64, 3, 2, 2, 1>;
using DecompressI8x128 = TcDecompressConfig<128, TACO_DI8_128_CFG / 1000, TACO_DI8_128_CFG / 100 % 10,
                                            TACO_DI8_128_CFG / 10 % 10, 1, TACO_DI8_128_CFG % 10>;
using DecompressI8x256 = TcDecompressConfig<256, 3, 2, 2, 1>;
using DecompressI8x512 = TcDecompressConfig<512, 3, 2, 2, 1>;

}  // namespace

KernelInfo decompress_kernel_info(int block, int code)
{
    if (code == 2) {
        switch (block) {
        case 64: return DecompressI8x64::info();
        case 128: return DecompressI8x128::info();
        case 256: return DecompressI8x256::info();
        case 512: return DecompressI8x512::info();
        default: return KernelInfo{};
        }
    }
    switch (block) {
    case 64: return DecompressTc64::info();
    case 128: return DecompressTc128::info();
    case 256: return DecompressTc256::info();
    case 512: return DecompressTc512::info();
    default: return KernelInfo{};
    }
}

cudaError_t launch_decompress(int block, Scheme scheme, const void *tmap_y, const void *packed, int64_t nblocks,
                              uint32_t *fault, int grid, cudaStream_t stream)
{
    const KernelInfo ki = decompress_kernel_info(block, scheme.code);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    CUtensorMap map;
    memcpy(&map, tmap_y, sizeof map);
    const uint8_t *pp = static_cast<const uint8_t *>(packed);
    void *args[] = {&map, &pp, &nblocks, &fault, &scheme};
    return launch_kernel(ki.fn, grid, ki.threads, ki.smem, stream, args);
}

}  // namespace taco
