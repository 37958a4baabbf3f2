// taco_compress.cu -- TACO's fused sender-side kernel (Algorithm 1, its
// compression loop; Eqs. 5-10) with the Hadamard rotation on the 5th-generation tensor
// cores (tcgen05), for GB300 (sm_103a).
//
// The rotation of a whole tile of blocks is a dense product: with the tile's
// 128 blocks as the rows of G (128 x B, bf16), Y = G H_B^T = G H_B (H_B is
// symmetric) holds y_k = H_B G_k in row k.  The products G_kj * (+-1) are exact
// and the tensor core accumulates in FP32, so Y is the unnormalised rotation
// of Eq. (8) up to FP32 summation order.  Blocks of 256 and 512 elements are
// 2 or 4 rows of 128 (tiles of 64 or 32 blocks): the MMA applies H_128 to each
// part and a butterfly across the parts' neighbouring TMEM lanes applies the
// H_2 or H_4 factor of H_B = H_2 (x) H_128 or H_4 (x) H_128.
//
// Scheduling: one CTA per tile of 128 rows, one CTA per SM resident; a
// running CTA takes its own tile, then the tiles of CTAs it cancels before
// they start (cluster launch control, taco_sched.cuh), so CTAs that get more
// memory bandwidth take more tiles and all SMs finish together.
//
// Roles in a CTA, one tile at a time:
//   warp 0  TMA producer: 2-D tiled loads (128-byte swizzle) of the tile into a
//           ring of STAGES shared-memory stages;
//   warp 1  allocates tensor memory and issues the tcgen05.mma of a tile
//           (M = 128, N = K = row length, BF16 in, FP32 out) into one of two to
//           four accumulators (tile i into accumulator i mod their number),
//           then commits to the stage's "empty" and the accumulator's "full"
//           barriers;
//   warps 2.. epilogue, EPG groups of 4 warps (group g takes every EPG-th
//           tile, so EPG tiles' epilogues can overlap): each thread
//           owns one row (one block or part) of the
//           accumulator in its TMEM lane: pass 1 reads it for the energy (by
//           Parseval, sum_j y_j^2 = B sum_j G_j^2) and the maximum, pass 2
//           reads it again and converts y * (Q_max / max|y|) to E4M3 two
//           codes at a time into a shared-memory record tile, which one
//           thread writes out with a bulk store.
// H_B is written once per CTA into shared memory in the same swizzled layout,
// by warps 1 and up while the CTA waits for the previous kernel.
//
// Scales: m = sum y^2 / B^2 (Eq. 6), alpha = tau / sqrt(m + eps) (Eq. 7),
// s = alpha * max|y| * (1/sqrt B) / Q_max (Eq. 9), codes of y * (Q_max / max|y|)
// (Eq. 10, alpha cancels); equal to the literal order up to FP32 rounding.
// Near zero (max|y| < 2^-100, where Q_max / max|y| can overflow) a warp codes
// its rows again from 2^64 y, which keeps the roundings of the unscaled
// formula.
//
// Ablations (Scheme): standard Hadamard + DS takes alpha = 1; DS only (its
// own instantiation, MODE 1) puts the identity in place of H (y = G) with
// alpha = 1 and codes G / s correctly rounded, as Eq. (10) writes it; ASH
// only stores s = 1 and converts Z = alpha y / sqrt(B) directly; E5M2 and
// INT8 codes use Q_max = 57344 and 127.  The rotating schemes with INT8 codes
// are their own instantiation too (MODE 2, scalar products before the integer
// rounding, see encode4_scaled), so the FP8 kernel carries no format branch
// around its packed products.
#include <cstring>
#include <type_traits>

#include <cuda.h>

#include "taco_device.cuh"
#include "taco_kernels.h"
#include "taco_sched.cuh"
#include "taco_tcgen05.cuh"

namespace taco {
namespace {


constexpr int kTcRows = 128;       // blocks per tile = MMA M = TMEM lanes
constexpr int kEpiThreads = 128;   // threads of one epilogue group (4 warps, one per TMEM lane part)

__host__ __device__ constexpr int tc_threads(int groups) { return 64 + kEpiThreads * groups; }

// B: block size; STAGES: A tiles in flight; EPG: epilogue groups (group g
// takes the tiles i with i % EPG == g, so EPG = 2 overlaps two tiles'
// epilogues); NBG: record-tile buffers per group.
template <int B, int STAGES, int EPG, int NBG>
struct TcCompressLayout {
    static constexpr int NOUT = EPG * NBG;                         // record-tile buffers
    // B = 256 and 512: each block is B / 128 A rows of 128 elements (its
    // parts), in neighbouring rows of the tile.
    static constexpr bool kSplit = B > 128;
    static constexpr int kRowElems = kSplit ? 128 : B;             // elements of an A row
    static constexpr int kRowsPerBlock = kSplit ? B / 128 : 1;
    static constexpr int kTileBlocks = kTcRows / kRowsPerBlock;    // blocks per tile
    static constexpr int kN = kRowElems;                           // MMA N = order of the Hadamard matrix used
    static constexpr int kKSteps = kN / 16;                        // MMAs (K = 16) per product with H_N
    static constexpr int kChunks = kRowElems / 64;                 // 128-byte K chunks of a row
    static constexpr int kChunkBytesA = kTcRows * 128;             // one chunk of the A tile
    static constexpr int kStageBytes = kTcRows * kRowElems * 2;    // one A tile
    static constexpr int kChunkBytesH = kN * 128;                  // one chunk of H_N
    static constexpr int kHBytes = kN * kN * 2;
    static constexpr int kRec = B + 8;
    static constexpr int kOutBytes = kTileBlocks * kRec;           // one record tile (multiple of 16)
    static constexpr int kAccCols = kRowElems;                     // TMEM columns of one accumulator
    // Accumulators in tensor memory (512 columns): up to four, so that more
    // than two epilogue groups can hold one each while the MMA fills the next.
    static constexpr int kNumAcc = 4 * kAccCols <= 512 ? 4 : 2;
    static constexpr int kTmemCols = kNumAcc * kAccCols;
    // Offsets from the 1024-byte aligned base.
    static constexpr int kOffA = 0;
    static constexpr int kOffH = kOffA + STAGES * kStageBytes;
    static constexpr int kOffOut = kOffH + kHBytes;
    // Tile scheduler.  The producer publishes item i after the empty barrier
    // of item i - STAGES, when the epilogues have read items up to
    // i - STAGES - 2: a published-tile slot (and the end marks of EPG items)
    // is reused only after every reader is done with it.
    static_assert(kTileRing >= STAGES + EPG + 2, "published-tile slot reused too early");
    static constexpr int kOffSched = kOffOut + NOUT * kOutBytes;   // 16-byte aligned
    static_assert(kOffSched % 16 == 0, "cancel responses need 16-byte alignment");
    static constexpr int kOffBar = kOffSched + kSchedBytes;        // 8-byte aligned
    static constexpr int kNumBars = 2 * STAGES + 2 * kNumAcc + 2 * NOUT;
    static constexpr int kOffTmem = kOffBar + 8 * kNumBars;
    static constexpr int kBytes = kOffTmem + 16;
    static constexpr int kSmem = kBytes + 1024;                    // slack for 1024-byte alignment
};

// Writes H_B (+-1 in bf16, Sylvester order; the identity when `rotate` is
// false) into shared memory as the K-major B operand in the 128-byte swizzled
// layout: chunk c holds columns [64c, 64c+64); row n of a chunk is 128 bytes
// whose 16-byte unit u sits at unit u ^ (n % 8).  Written by the threads of
// warps 1 and up, before their dependency wait: warp 0's thread 0 issues the
// first loads right after that wait and would otherwise hold the CTA's set-up
// barrier for its share (about 0.5 us for one thread alone).
template <int B>
__device__ void write_hadamard_sw128(uint8_t *h, bool rotate)
{
    constexpr int kUnits = B * (B / 8);    // 16-byte units of H
    if (threadIdx.x < 32)
        return;
    for (int idx = threadIdx.x - 32; idx < kUnits; idx += blockDim.x - 32) {
        const int n = idx / (B / 8);
        const int u_all = idx % (B / 8);   // unit index along K over the whole row
        const int c = u_all / 8, u = u_all % 8;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int k0 = 8 * u_all + 2 * q;
            uint32_t lo = (__popc(n & k0) & 1) ? 0xBF80u : 0x3F80u;
            uint32_t hi = (__popc(n & (k0 + 1)) & 1) ? 0xBF80u : 0x3F80u;
            if (!rotate) {
                lo = (n == k0) ? 0x3F80u : 0u;
                hi = (n == k0 + 1) ? 0x3F80u : 0u;
            }
            w[q] = lo | (hi << 16);
        }
        uint8_t *dst = h + c * (B * 128) + n * 128 + ((u ^ (n & 7)) * 16);
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// MODE: 0 rotation, FP8 codes (E4M3 or E5M2); 1 DS only, any code format;
// 2 rotation, INT8 codes.
template <int B, int STAGES, int EPG, int NBG, int MODE>
__global__ void __launch_bounds__(tc_threads(EPG), 1)
    taco_compress_kernel(const __grid_constant__ CUtensorMap tmap_x, uint8_t *__restrict__ packed,
                            int64_t nblocks, uint32_t *__restrict__ fault, const Scheme scheme)
{
    using Lay = TcCompressLayout<B, STAGES, EPG, NBG>;
    constexpr int NOUT = Lay::NOUT;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(base);
    const uint32_t bar0 = sbase + Lay::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    constexpr int NACC = Lay::kNumAcc;
    auto acc_full_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto acc_empty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + NACC + a); };
    auto out_free_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * NACC + b); };
    auto rec_done_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * NACC + NOUT + b); };
    const TileSched sched{sbase + Lay::kOffSched, fault, kFaultCompress};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + Lay::kOffTmem);

    grid_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- set-up ----------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NACC; a++) {
            mbar_init(acc_full_bar(a), 1);
            mbar_init(acc_empty_bar(a), kEpiThreads / 32);   // the 4 warps of the group reading it
        }
        for (int b = 0; b < NOUT; b++) {
            mbar_init(out_free_bar(b), 1);
            mbar_init(rec_done_bar(b), kEpiThreads / 32);
        }
        sched.init();
        fence_mbar_init();
        prefetch_tmap(&tmap_x);
    }
    // The producer (thread 0) sends the first kSchedAhead tile requests and
    // starts its own tile's load (item 0) before the rest of the set-up.
    auto issue_tile = [&](int i, int64_t t) {
        const int s = i % STAGES;
        mbar_arrive_expect_tx(full_bar(s), Lay::kStageBytes);
        const uint32_t dst = sbase + Lay::kOffA + s * Lay::kStageBytes;
#pragma unroll
        for (int c = 0; c < Lay::kChunks; c++)
            tma_load_2d(dst + c * Lay::kChunkBytesA, &tmap_x, 64 * c, static_cast<int32_t>(t * kTcRows), full_bar(s));
    };
    if (threadIdx.x == 0) {
        for (int j = 1; j <= kSchedAhead; j++)
            sched.request(j);
        // While the previous kernel drains: its own tile and, as a guess at
        // the tiles of the next rounds, those one and more SM counts further on.
        for (int k = 0; k < kL2PrefetchCompress; k++) {
            const uint32_t t = blockIdx.x + k * num_sms();
            if (t < gridDim.x)
#pragma unroll
                for (int c = 0; c < Lay::kChunks; c++)
                    tma_prefetch_2d(&tmap_x, 64 * c, static_cast<int32_t>(t * kTcRows));
        }
        grid_dependency_wait();   // the input may come from the previous kernel
        sched.publish(0, blockIdx.x);
        issue_tile(0, blockIdx.x);
    }
    if (warp == 1)
        tmem_alloc(smem_addr(tmem_slot), Lay::kTmemCols);
    // DS only (no rotation) is its own instantiation; the others rotate.
    constexpr bool DS_ONLY = MODE == 1;
    constexpr bool rotate = !DS_ONLY;
    const bool adaptive = scheme.variant == 0 || scheme.variant == 3;  // alpha from Eqs. (6)-(7)
    const bool dual_scale = scheme.variant != 3;                    // s from Eq. (9)
    write_hadamard_sw128<Lay::kN>(base + Lay::kOffH, rotate);
    fence_proxy_async_smem();   // H is read by the tensor core (async proxy)
    tc_fence_before_sync();
    grid_dependency_wait();   // before any global access of this thread
    cta_barrier();   // lanes of warps 0 and 1 took different paths above
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---- TMA producer ------------------------------------------------
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
                const int s = i % STAGES;
                if (i >= STAGES &&
                    !mbar_wait_bounded_thread(empty_bar(s), ((i / STAGES) - 1) & 1, fault, kFaultCompress)) {
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
            for (int j = issued - STAGES > 0 ? issued - STAGES : 0; j < issued; j++)
                mbar_wait_bounded_thread(full_bar(j % STAGES), (j / STAGES) & 1, fault, kFaultCompress);
        }
    } else if (warp == 1) {
        // ---- MMA issuer --------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = mma_idesc_bf16_f32(kTcRows, Lay::kN);
            const uint32_t a0 = sbase + Lay::kOffA, h0 = sbase + Lay::kOffH;
            int i = 0;
            for (;; i++) {
                if (sched.tile_thread(i) < 0)
                    break;
                const int s = i % STAGES, acc = i % NACC;
                if (i >= NACC && !mbar_wait_bounded_thread(acc_empty_bar(acc), ((i / NACC) - 1) & 1, fault,
                                                        kFaultCompress))
                    break;
                if (!mbar_wait_bounded_thread(full_bar(s), (i / STAGES) & 1, fault, kFaultCompress))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * Lay::kAccCols);
                const uint32_t a_stage = a0 + s * Lay::kStageBytes;
#pragma unroll
                for (int kk = 0; kk < Lay::kKSteps; kk++) {
                    const uint32_t koff = (kk & 3) * 32;   // 16 bf16 = 32 bytes along K
                    const uint64_t ad = sw128_kmajor_desc(a_stage + (kk >> 2) * Lay::kChunkBytesA + koff);
                    const uint64_t bd = sw128_kmajor_desc(h0 + (kk >> 2) * Lay::kChunkBytesH + koff);
                    tc_mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(empty_bar(s));
                tc_commit(acc_full_bar(acc));
            }
            // All MMAs issued must finish before tensor memory is freed.
            if (i > 0)
                mbar_wait_bounded_thread(acc_full_bar((i - 1) % NACC), ((i - 1) / NACC) & 1, fault, kFaultCompress);
        }
    } else {
        // ---- epilogue (warps 2 .. 2+4*EPG-1) --------------------------------
        const int grp = (warp - 2) / 4;                 // epilogue group
        const int et = threadIdx.x - 64 - kEpiThreads * grp;   // 0..127 within the group
        const int q = warp & 3;                         // TMEM lane part of this warp
        const int row = 32 * q + lane;                  // accumulator row
        const int blk = row / Lay::kRowsPerBlock;       // block within the tile
        const int part = row % Lay::kRowsPerBlock;      // B = 256 / 512: which 128 elements of the block
        const bool store_warp = ((warp - 2) & 3) == 0;  // first warp of the group issues the stores
        const float rB = (B == 64)    ? 0.125f
                         : (B == 128) ? 0.0883883476483184405f
                         : (B == 256) ? 0.0625f
                                      : 0.0441941738241592203f;   // 1/sqrt(B) in binary32
        for (int kt = 0;; kt++) {                   // kt: tiles this group has handled
            const int i = EPG * kt + grp;               // the CTA's item counter
            const int64_t t = sched.tile_warp(i);
            if (t < 0)
                break;
            const int acc = i % NACC;
            if (!mbar_wait_bounded(acc_full_bar(acc), (i / NACC) & 1, fault, kFaultCompress))
                break;
            tc_fence_after_sync();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * Lay::kAccCols);

            // Pass 1: energy (Parseval) and max|y|.
            float2 e2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            float ymax = 0.f;
            // B = 256 / 512: H_B = H_2 (x) H_128 / H_4 (x) H_128 (Sylvester
            // order); the MMA gave H_128 of each part, the parts' rows sit in
            // neighbouring lanes, and a butterfly over lanes (xor 1; and xor 2
            // for four parts) finishes the rotation.  The rotated part goes
            // back into its TMEM columns; pass 2 reads it from there, as for
            // the other block sizes.
            if constexpr (Lay::kSplit) {
                const float sgn1 = (part & 1) ? -1.0f : 1.0f, sgn2 = (part & 2) ? -1.0f : 1.0f;
#pragma unroll 1
                for (int c = 0; c < 4; c++) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 32 * c, r);
                    tmem_ld_wait();
                    tmem_regs_ready(r);
#pragma unroll
                    for (int j = 0; j < 32; j++) {
                        float v = __uint_as_float(r[j]);
                        if (rotate) {   // lower lane a + b, upper lane a - b, as one fma each
                            v = fmaf(sgn1, v, __shfl_xor_sync(kFullMask, v, 1));
                            if constexpr (Lay::kRowsPerBlock == 4)
                                v = fmaf(sgn2, v, __shfl_xor_sync(kFullMask, v, 2));
                        }
                        r[j] = __float_as_uint(v);
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 y = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                        e2[(j >> 1) & 3] = fma2(y, y, e2[(j >> 1) & 3]);
                        ymax = max3(ymax, fabsf(y.x), fabsf(y.y));
                    }
                    if (rotate)
                        tmem_st32(taddr + 32 * c, r);
                }
                tmem_st_wait();
            } else {
#pragma unroll
                for (int c = 0; c < B / 32; c++) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 32 * c, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 y = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                        e2[(j >> 1) & 3] = fma2(y, y, e2[(j >> 1) & 3]);
                        ymax = max3(ymax, fabsf(y.x), fabsf(y.y));
                    }
                }
            }
            const float2 e01 = add2(e2[0], e2[1]), e23 = add2(e2[2], e2[3]);
            const float2 ee = add2(e01, e23);
            float etot = ee.x + ee.y;
#pragma unroll
            for (int d = 1; d < Lay::kRowsPerBlock; d <<= 1) {   // over the block's parts
                etot += __shfl_xor_sync(kFullMask, etot, d);
                ymax = fmaxf(ymax, __shfl_xor_sync(kFullMask, ymax, d));
            }
            const float m = etot * (1.0f / (static_cast<float>(B) * B));
            const float alpha = adaptive ? __fdiv_rn(kTau, __fsqrt_rn(m + kEps)) : 1.0f;
            const float rr = rotate ? rB : 1.0f;
            const float qmax = code_qmax(scheme.code);
            float s = 0.f, k = 0.f;
            if (!dual_scale) {            // ASH only: codes of Z = alpha r y, s = 1
                s = 1.0f;
                k = __fmul_rn(alpha, rr);
            } else if (ymax > 0.f) {
                s = __fdiv_rn(__fmul_rn(__fmul_rn(alpha, ymax), rr), qmax);
                k = __fdiv_rn(qmax, ymax);
            }

            // The group's record tile buffer used NBG tiles ago must have been read
            // by its bulk store before it is overwritten: thread 0 (which
            // issued that store) confirms it on out_free, the others wait.
            const int ob = grp * NBG + (kt % NBG);
            if (kt >= NBG) {
                if (et == 0) {
                    bulk_wait_read<NBG - 1>();
                    mbar_arrive(out_free_bar(ob));
                }
                if (!mbar_wait_bounded(out_free_bar(ob), ((kt / NBG) - 1) & 1, fault, kFaultCompress))
                    break;
            }
            const uint32_t rec_block = sbase + Lay::kOffOut + ob * Lay::kOutBytes + blk * Lay::kRec;
            const uint32_t rec = rec_block + part * 128;

            const float srcp = DS_ONLY ? __frcp_rn(s) : 0.f;   // DS only: 1/s, correctly rounded
            // Pass 2: codes (Eq. 10) two per cvt, 32 per chunk.  `scaled`:
            // every value is first multiplied by `pre` (exact).
            auto code_pass = [&](float kk, auto scaled, float pre) {
                // The rare scaled pass and DS only stay compact (one chunk at
                // a time).
#pragma unroll((decltype(scaled)::value || DS_ONLY) ? 1 : Lay::kAccCols / 32)
                for (int c = 0; c < Lay::kAccCols / 32; c++) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 32 * c, r);
                    tmem_ld_wait();
                    if constexpr (decltype(scaled)::value) {
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), pre));
                    }
                    uint32_t cw[8];
                    if constexpr (MODE == 2) {
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            cw[j] = encode4_scaled(
                                2, make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])),
                                make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), kk);
                    } else if constexpr (MODE == 0) {
                        const float2 k2 = make_float2(kk, kk);
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            const float2 u0 =
                                mul2(make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])), k2);
                            const float2 u1 =
                                mul2(make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), k2);
                            cw[j] = encode4(scheme.code, u0.x, u0.y, u1.x, u1.y);
                        }
                    } else if (s >= kDivFastMin) {
                        // DS only: the unrotated block's values G / s with s =
                        // max|G| / Q_max, correctly rounded as Eq. (10) writes it
                        // (ratios of bf16 values land exactly on rounding
                        // midpoints often, and there only the quotient itself
                        // decides the code as the method does).
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            const float2 u0 = div2_by(
                                make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])), s, srcp);
                            const float2 u1 = div2_by(
                                make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), s, srcp);
                            cw[j] = encode4(scheme.code, u0.x, u0.y, u1.x, u1.y);
                        }
                    } else {
                        // DS only with a tiny (or zero) s: IEEE division.
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            float u[4];
#pragma unroll
                            for (int h = 0; h < 4; h++)
                                u[h] = s > 0.f ? __fdiv_rn(__uint_as_float(r[4 * j + h]), s) : 0.f;
                            cw[j] = encode4(scheme.code, u[0], u[1], u[2], u[3]);
                        }
                    }
                    if (!(ymax > 0.f)) {
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            cw[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        sts64(rec + 32 * c + 8 * j, cw[2 * j], cw[2 * j + 1]);
                }
            };
            code_pass(k, std::false_type{}, 1.0f);
            if constexpr (!DS_ONLY) {
                // A tiny rotation (0 < max|y| < 2^-100; Q_max / max|y| may
                // have overflowed above) is coded again from values scaled by
                // 2^64, which keeps the roundings of the unscaled formula.  DS
                // only divides and needs no scaling.
                const bool tiny = dual_scale && ymax > 0.f && ymax < kTinyValue;
                if (__any_sync(kFullMask, tiny)) {     // warp-uniform, rare
                    const float pre = tiny ? kTinyUp : 1.0f;
                    code_pass(__fdiv_rn(qmax, __fmul_rn(ymax, pre)), std::true_type{}, pre);
                }
            }
            // The accumulator is read: hand it back to the MMA warp.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acc_empty_bar(acc));

            if (part == 0)
                sts64(rec_block + B, __float_as_uint(alpha), __float_as_uint(s));
            fence_proxy_async_smem();
            __syncwarp();                               // one arrival per warp covers its lanes' writes
            if (lane == 0)
                mbar_arrive(rec_done_bar(ob));

            // The group's first warp (lane 0) stores the tile's records once all are written.
            constexpr int TB = Lay::kTileBlocks;
            const int64_t blk0 = t * TB;
            const int nvalid = static_cast<int>(nblocks - blk0 < TB ? nblocks - blk0 : TB);
            const int neven = nvalid & ~1;
            if (store_warp) {
                if (!mbar_wait_bounded(rec_done_bar(ob), (kt / NBG) & 1, fault, kFaultCompress))
                    break;
                if (lane == 0 && neven > 0) {
                    bulk_store(packed + blk0 * Lay::kRec, sbase + Lay::kOffOut + ob * Lay::kOutBytes,
                               static_cast<uint32_t>(neven * Lay::kRec));
                    bulk_commit();
                }
            }
            if ((nvalid & 1) && blk == nvalid - 1 && part == 0) {
                uint8_t *dst = packed + (blk0 + blk) * Lay::kRec;
                const uint8_t *src = base + Lay::kOffOut + ob * Lay::kOutBytes + blk * Lay::kRec;
                for (int o = 0; o < Lay::kRec; o += 8)
                    *reinterpret_cast<uint2 *>(dst + o) = *reinterpret_cast<const uint2 *>(src + o);
            }
        }
        // The shared-memory sources of this thread's stores must be read
        // before the CTA exits; the writes themselves complete before the
        // grid does.
        if (et == 0)
            bulk_wait_read<0>();
    }

    // ---- tear-down -------------------------------------------------------
    tc_fence_before_sync();
    cta_barrier();   // every role ran lane-divergent code
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Lay::kTmemCols);
    }
}

template <int B, int STAGES, int EPG, int NBG>
struct TcCompressConfig {
    using Lay = TcCompressLayout<B, STAGES, EPG, NBG>;
    static_assert(Lay::kSmem <= 227 * 1024, "shared memory budget");
    static void *fn(int mode)
    {
        return mode == 1   ? reinterpret_cast<void *>(&taco_compress_kernel<B, STAGES, EPG, NBG, 1>)
               : mode == 2 ? reinterpret_cast<void *>(&taco_compress_kernel<B, STAGES, EPG, NBG, 2>)
                           : reinterpret_cast<void *>(&taco_compress_kernel<B, STAGES, EPG, NBG, 0>);
    }
    static KernelInfo info(int mode)
    {
        return KernelInfo{fn(mode), static_cast<size_t>(Lay::kSmem), tc_threads(EPG), Lay::kTileBlocks, 0};
    }
};

#ifndef TACO_TC64_CFG
#define TACO_TC64_CFG 641
#endif
#ifndef TACO_TC128_CFG
#define TACO_TC128_CFG 431
#endif
#ifndef TACO_TC256_CFG
#define TACO_TC256_CFG 331
#endif
#ifndef TACO_TC512_CFG
#define TACO_TC512_CFG 341
#endif
// Per block size, three digits: A stages, epilogue groups, buffers per group.
using CompressTc64 = TcCompressConfig<64, TACO_TC64_CFG / 100, TACO_TC64_CFG / 10 % 10, TACO_TC64_CFG % 10>;
using CompressTc128 = TcCompressConfig<128, TACO_TC128_CFG / 100, TACO_TC128_CFG / 10 % 10, TACO_TC128_CFG % 10>;
using CompressTc256 = TcCompressConfig<256, TACO_TC256_CFG / 100, TACO_TC256_CFG / 10 % 10, TACO_TC256_CFG % 10>;
using CompressTc512 = TcCompressConfig<512, TACO_TC512_CFG / 100, TACO_TC512_CFG / 10 % 10, TACO_TC512_CFG % 10>;

}  // namespace

KernelInfo compress_kernel_info(int block, int variant, int code)
{
    const int mode = variant == 2 ? 1 : code == 2 ? 2 : 0;
    switch (block) {
    case 64: return CompressTc64::info(mode);
    case 128: return CompressTc128::info(mode);
    case 256: return CompressTc256::info(mode);
    case 512: return CompressTc512::info(mode);
    default: return KernelInfo{};
    }
}

cudaError_t launch_compress(int block, Scheme scheme, const void *tmap, void *packed, int64_t nblocks, uint32_t *fault,
                            int grid, cudaStream_t stream)
{
    const KernelInfo ki = compress_kernel_info(block, scheme.variant, scheme.code);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    CUtensorMap map;
    memcpy(&map, tmap, sizeof map);
    uint8_t *pp = static_cast<uint8_t *>(packed);
    void *args[] = {&map, &pp, &nblocks, &fault, &scheme};
    return launch_kernel(ki.fn, grid, ki.threads, ki.smem, stream, args);
}

}  // namespace taco
