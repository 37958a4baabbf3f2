// taco_reduce.cu -- receive-side local reduction of TACO's two-shot compressed
// AllReduce (Section 4.4.2: a compressed all-to-all exchange, then one
// reduction per owner) for GB300 (sm_103a): P packed shards in local HBM
// are decoded to FP32, summed, and the sum is compressed once.
//
// No rotation is needed.  Shard p decodes to G'_p = R (q_p s_p / alpha_p) with
// R = (1/sqrt B) H_B, and R is symmetric and orthogonal (R R = I).  For the sum
// S = R W with W = sum_p q_p (s_p / alpha_p); compressing S gives
// mean(S^2) = |W|^2 / B, Z = alpha' R S = alpha' W, s' = alpha' max|W| / Q_max and
// codes Cvt_FP8(Q_max W / max|W|).  The kernel computes exactly these, which
// differ from decode-sum-encode with explicit rotations only by FP32 rounding.
// Near zero (a block sum below 2^-80, where the factors s_p / alpha_p are
// subnormal or zero in binary32) the block is summed again from global memory
// with factors 2^64 s_p / alpha_p and its scales taken back by 2^-64.  DS only
// has no rotation: W is the FP32 sum of the decoded shards itself, coded as
// W / s' correctly rounded.
//
// Data movement.  A tile is T consecutive blocks (T = 4096 / B for most shard
// counts; twice that for the 4-shard kernel, four times for the 2-shard
// kernel, which takes two passes per tile, and half of it for the 16-shard
// kernel at B = 32); its records are contiguous in every shard, T * (B + 8)
// bytes (a multiple of 16: T is even).  The loader warp bulk-copies the
// tile's P record runs (lane p the run of shard p) into one stage of a
// shared-memory ring (as many stages of P runs as fit in its 192 KB; the
// 16-shard kernel's ring holds exactly three stages) and a group of 8
// consumer warps decodes them from shared memory (three groups take turns, so
// three tiles are decoded at once): each thread owns LC consecutive elements
// of a block (16; 32 in the 2- and 4-shard kernels; TACO_REDUCE_LANE_CODES = 8
// halves the 16 where a block still fits a warp, measured slower), so B / LC
// consecutive threads share a block.  Energy and maximum are reduced across
// the block's threads with xor-shuffles (every thread ends with the same
// bits), and every thread stores its codes directly (8-byte stores).
//
// Ablations: the decode of every code format is exact (E4M3 and E5M2 through
// f16, INT8 as integers), W is the same for every variant, and the output
// takes alpha' = 1 for standard Hadamard + DS and DS only (s' = max|W| / Q_max),
// or s' = 1 and codes Cvt(alpha' W) for ASH only.
//
// Scheduling: one CTA per tile, one CTA per SM resident (shared memory); the
// resident CTA takes its own tile, then the tiles of CTAs it cancels before
// they start (cluster launch control, taco_sched.cuh).  The loader publishes a
// tile to the consumers only when it issues its copies, after the stage's
// previous item was released, so the consumer groups, which take turns on the
// stages, never see an older phase of a stage barrier as the one they wait for.
#include <type_traits>

#include "taco_device.cuh"
#include "taco_kernels.h"
#include "taco_sched.cuh"
#include "taco_tcgen05.cuh"

namespace taco {
namespace {

#ifndef TACO_REDUCE_RING_KB
#define TACO_REDUCE_RING_KB 192
#endif
#ifndef TACO_REDUCE_FIXED_SHARDS
#define TACO_REDUCE_FIXED_SHARDS 1
#endif
#ifndef TACO_REDUCE_GROUPS
#define TACO_REDUCE_GROUPS 3
#endif
#ifndef TACO_REDUCE_CONSUMERS
#define TACO_REDUCE_CONSUMERS 256
#endif
constexpr int kConsumers = TACO_REDUCE_CONSUMERS;   // threads of a consumer group
constexpr int kGroups = TACO_REDUCE_GROUPS;     // consumer groups; group g takes items i % kGroups == g
constexpr int kRThreads = kGroups * kConsumers + 32;   // + the loader warp
#ifndef TACO_REDUCE_LANE_CODES
#define TACO_REDUCE_LANE_CODES 16
#endif
constexpr int kLaneCodes = TACO_REDUCE_LANE_CODES;   // codes (elements) per thread per shard
static_assert(kLaneCodes == 8 || kLaneCodes == 16, "8 or 16 codes per thread");
constexpr int kRingBytes = TACO_REDUCE_RING_KB * 1024;
constexpr int kMaxStages = 8;
#ifndef TACO_REDUCE_SCHED_AHEAD
#define TACO_REDUCE_SCHED_AHEAD TACO_SCHED_AHEAD
#endif
constexpr int kRSchedAhead = TACO_REDUCE_SCHED_AHEAD;   // cancel requests in flight
// The loader publishes item i after the empty barrier of item i - nst, when
// the consumers have read every item up to i - nst: a published-tile slot
// (and the end marks of kGroups items) is reused only after its readers are done.
static_assert(kTileRing >= kMaxStages + kGroups, "published-tile slot reused too early");

// MUL: passes of the consumer group over a tile.  The 2-shard kernel takes
// tiles of two passes, so that a stage still holds about 35 KB of records in
// long runs (the copies of 2 shards at the 8-shard tile size moved 42% of the
// bandwidth).
// LCODES: codes per thread per shard (0: kLaneCodes).  The 2- and 4-shard
// kernels give each thread 32: with few shards a thread's work is mostly the
// per-block epilogue (energy, maximum, scales, conversion, stores), which it
// then does once for twice the codes (16384 x 8192: 2 shards 42.1 -> 34.5 us,
// 4 shards 30.4 -> 27.4 us; 32 codes at 8 shards were slower, 25.6 -> 26.7 us).
// MAXP: the shard count the layout is sized for (0: from MUL).
// RING: bytes of the stage ring.  The 16-shard and the generic kernels for
// B >= 64 size it for exactly three stages of 16 runs of full tiles
// (195-216 KB): two stages, or tiles halved to 8 codes per thread (2.2 KB
// copies, five stages), kept DRAM under-fed (16384 x 8192, 16 shards:
// 31.4 -> 24.8 us).  B = 32 would fit only two such stages: its 16-shard
// kernel keeps halved tiles, its generic kernel the 192 KB ring.
template <int B, int MUL = 1, int LCODES = 0, int RING = kRingBytes, int MAXP = 0>
struct ReduceLayout {
    // Codes per thread: LCODES or kLaneCodes, or 16 where a block would span
    // more than a warp (its energy and maximum are reduced with shuffles inside
    // one warp).
    static constexpr int kLC0 = LCODES > 0 ? LCODES : kLaneCodes;
    static constexpr int kLC = B / kLC0 > 32 ? 16 : kLC0;
    static constexpr int kLW = kLC / 4;                      // 32-bit words of a thread's codes
    // Shards a kernel of this layout takes at most.
    static constexpr int kMaxP = MAXP > 0 ? MAXP : MUL > 1 ? 8 / MUL : kMaxShards;
    // Blocks per consumer pass: one per kLpb consumer threads, halved until two
    // stages of kMaxP record runs of a tile fit the ring (the threads beyond it
    // stay idle).
    static constexpr int pass_blocks()
    {
        int t = kConsumers * kLC / B;
        while (t > 2 && 2 * kMaxP * MUL * t * (B + 8) > RING)
            t /= 2;
        return t;
    }
    static constexpr int kSub = pass_blocks();
    static constexpr int kT = MUL * kSub;                    // blocks per tile
    static constexpr int kLpb = B / kLC;                     // threads per block
    static_assert(kLpb <= 32 && 32 % kLpb == 0, "a block's threads lie in one warp");
    static constexpr int kRec = B + 8;
    static constexpr int kRunBytes = kT * kRec;             // one shard's records of a tile
    static_assert(kT % 2 == 0 && kRunBytes % 16 == 0, "bulk copies need 16-byte multiples");
    static constexpr int kRing = RING;
    static_assert(kRing >= 2 * kMaxP * kRunBytes, "at least two stages at the largest shard count");
    // Offsets from the 128-byte aligned base.
    static constexpr int kOffRing = 0;
    static constexpr int kOffSched = kOffRing + kRing;                // 16-byte aligned
    static constexpr int kOffPtrs = kOffSched + kSchedBytes;
    static constexpr int kOffBar = kOffPtrs + 8 * kMaxShards;
    static constexpr int kNumBars = 2 * kMaxStages;
    static constexpr int kBytes = kOffBar + 8 * kNumBars;
    static constexpr int kSmem = kBytes + 128;                        // slack for alignment
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// The layout of the reduce kernel for block B, code format CODE and shard
// count PFIX (0: any count; -4: any count up to 4, which takes the 2- and
// 4-shard kernels' 32 codes per thread).
__host__ __device__ constexpr int reduce_mul(int pfix) { return pfix == 2 ? 2 : 1; }
__host__ __device__ constexpr int reduce_lcodes(int B, int pfix)
{
    return pfix == 2 || pfix == 4 || pfix == -4 ? 32 : pfix == 16 && B < 64 ? 8 : 0;
}
__host__ __device__ constexpr int reduce_maxp(int pfix) { return pfix < 0 ? -pfix : pfix; }
__host__ __device__ constexpr int reduce_ring(int B, int pfix)
{
    return (pfix == 16 || pfix == 0) && B >= 64 ? 3 * 16 * (kConsumers * 16 / B) * (B + 8) : kRingBytes;
}
template <int B, int PFIX>
using ReduceLayoutFor =
    ReduceLayout<B, reduce_mul(PFIX), reduce_lcodes(B, PFIX), reduce_ring(B, PFIX), reduce_maxp(PFIX)>;

// Values of the four codes in `x`, first code in .x of the first pair.
template <int CODE>
__device__ __forceinline__ void decode4(uint32_t x, float2 &q0, float2 &q1)
{
    if constexpr (CODE == 0) {
        q0 = e4m3x2_to_float2(x & 0xffffu);
        q1 = e4m3x2_to_float2(x >> 16);
    } else if constexpr (CODE == 1) {
        // An E5M2 code is the high byte of the f16 of the same value
        // (subnormals and signs included): byte permutes build both f16 pairs.
        q0 = f16x2_to_float2(__byte_perm(x, 0u, 0x1404));
        q1 = f16x2_to_float2(__byte_perm(x, 0u, 0x3424));
    } else {
        int8x4_to_float(x, q0, q1);
    }
}

// w[k] += q[k] * f for the thread's codes in `words`, each product rounded on
// its own before the add (so that a shard and its negation cancel exactly, as
// in an FP32 sum of decoded shards).  The products stay scalar: packed ones
// (__fmul2_rn, mul.rn.f32x2, or fma.rn.f32x2 with a -0 addend) before the
// packed add came out fused into FFMA2, which tests/test_gpu_reduce_exact_sum.py
// detects.
template <int CODE, int LW>
__device__ __forceinline__ void accumulate_shard(float (&w)[4 * LW], const uint32_t (&words)[LW], float f)
{
#pragma unroll
    for (int k = 0; k < LW; k++) {
        float2 q0, q1;
        decode4<CODE>(words[k], q0, q1);
        // Scalar products (never contracted), packed sums.
        const float2 t0 = make_float2(__fmul_rn(q0.x, f), __fmul_rn(q0.y, f));
        const float2 t1 = make_float2(__fmul_rn(q1.x, f), __fmul_rn(q1.y, f));
        const float2 s0 = add2(make_float2(w[4 * k + 0], w[4 * k + 1]), t0);
        const float2 s1 = add2(make_float2(w[4 * k + 2], w[4 * k + 3]), t1);
        w[4 * k + 0] = s0.x;
        w[4 * k + 1] = s0.y;
        w[4 * k + 2] = s1.x;
        w[4 * k + 3] = s1.y;
    }
}

__device__ __forceinline__ uint2 ldg_u2(const uint8_t *p)
{
    return *reinterpret_cast<const uint2 *>(p);
}

// PFIX > 0: the shard count is fixed at compile time (the shard loop unrolls);
// 0 or -4: the count is the call's (any, or at most 4).
template <int B, int CODE, int PFIX>
__global__ void __launch_bounds__(kRThreads, 1) taco_shard_reduce_kernel(const ReduceArgs args, uint32_t *fault)
{
    constexpr int MUL = reduce_mul(PFIX);
    using Lay = ReduceLayoutFor<B, PFIX>;
    constexpr int T = Lay::kT;
    constexpr int kRec = Lay::kRec;
    constexpr int LC = Lay::kLC, LW = Lay::kLW;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *base = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
    const uint32_t sbase = smem_addr(base);
    const uint32_t bar0 = sbase + Lay::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    const TileSched sched{sbase + Lay::kOffSched, fault, kFaultReduce};
    const uint8_t **shard_ptr = reinterpret_cast<const uint8_t **>(base + Lay::kOffPtrs);

    grid_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int P = PFIX > 0 ? PFIX : args.num_shards;
    const int64_t nblocks = args.nblocks;
    const bool adaptive = args.variant == 0 || args.variant == 3;   // alpha' from the energy of W
    const bool dual_scale = args.variant != 3;                      // s' from max|W|
    const bool ds_only = args.variant == 2;                         // no rotation: W is the decoded sum
    // Stages of P record runs in the ring.
    const int stage_bytes = P * Lay::kRunBytes;
    int nst = Lay::kRing / stage_bytes;
    nst = nst > kMaxStages ? kMaxStages : nst;

    auto tile_valid = [&](int64_t t) {
        const int64_t left = nblocks - t * T;
        return static_cast<int>(left < T ? left : T);
    };

    // ---- set-up ----------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumers / 32);
        }
        sched.init();
        fence_mbar_init();
    }
    if (threadIdx.x < kMaxShards)
        shard_ptr[threadIdx.x] = args.shards[threadIdx.x];
    if (warp == kGroups * kConsumers / 32 && lane < P) {
        // While the previous kernel drains: this CTA's tile of shard `lane`
        // and, as a guess at the next rounds' tiles, one and more SM counts on.
        for (int k = 0; k < kL2PrefetchReduce; k++) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(k) * num_sms();
            if (t < gridDim.x) {
                const uint32_t run = static_cast<uint32_t>(tile_valid(t) & ~1) * kRec;   // multiple of 16
                if (run > 0)
                    bulk_prefetch_l2(args.shards[lane] + t * T * kRec, run);
            }
        }
    }
    grid_dependency_wait();   // the shards may come from the previous kernel
    cta_barrier();

    if (warp == kGroups * kConsumers / 32) {
        // ---- loader: lane 0 runs the tile scheduler and the stage barriers,
        // lane p issues the bulk copy of shard p (the copies of a tile go out
        // at once instead of one after another from one thread).
        auto issue_tile = [&](int i, int64_t t) {   // whole warp
            const int s = i % nst;
            const int nvalid = tile_valid(t);
            const uint32_t run = static_cast<uint32_t>(nvalid & ~1) * kRec;   // multiple of 16
            if (lane == 0)
                mbar_arrive_expect_tx(full_bar(s), run * static_cast<uint32_t>(P));
            __syncwarp();
            if (run > 0 && lane < P)
                bulk_load(sbase + Lay::kOffRing + s * stage_bytes + lane * Lay::kRunBytes,
                          shard_ptr[lane] + t * T * kRec, run, full_bar(s));
        };
        int requested = kRSchedAhead;   // requests 1 .. requested issued (lane 0)
        if (lane == 0) {
            for (int j = 1; j <= kRSchedAhead; j++)
                sched.request(j);
            sched.publish(0, blockIdx.x);
        }
        issue_tile(0, blockIdx.x);
        int i = 1;                       // items 0 .. i-1 have been loaded
        for (;; i++) {
            int64_t t = -1;
            if (lane == 0) {
                t = sched.response(i);
                if (t >= 0) {
                    sched.request(++requested);  // no failure seen yet: keep kRSchedAhead in flight
                    const int s = i % nst;
                    if (i >= nst &&
                        !mbar_wait_bounded_thread(empty_bar(s), ((i / nst) - 1) & 1, fault, kFaultReduce))
                        t = -1;
                }
                if (t < 0)
                    sched.publish_end(i, kGroups);
                else
                    sched.publish(i, t);
            }
            t = __shfl_sync(kFullMask, t, 0);
            if (t < 0)
                break;
            issue_tile(i, t);
        }
        // Responses still in flight and the tile copies must land before the
        // CTA can exit.
        if (lane == 0) {
            sched.drain(i, requested);
            for (int j = i - nst > 0 ? i - nst : 0; j < i; j++)
                mbar_wait_bounded_thread(full_bar(j % nst), (j / nst) & 1, fault, kFaultReduce);
        }
    } else {
        // ---- consumers: Lay::kLC elements of one block per thread ------------
        const int grp = threadIdx.x / kConsumers;
        const int c = threadIdx.x % kConsumers;
        const int bl = c / Lay::kLpb;        // block within the tile
        const int part = c % Lay::kLpb;      // Lay::kLC-element part of the block
        for (int i = grp;; i += kGroups) {
            const int64_t t = sched.tile_warp(i);
            if (t < 0)
                break;
            const int s = i % nst;
            if (!mbar_wait_bounded(full_bar(s), (i / nst) & 1, fault, kFaultReduce))
                break;
            const int nvalid = tile_valid(t);
#pragma unroll 1
            for (int sub = 0; sub < MUL; sub++) {
            const int blt = sub * Lay::kSub + bl;                          // block within the tile
            const bool active = bl < Lay::kSub && blt < nvalid;
            const bool from_global = (nvalid & 1) && blt == nvalid - 1;   // not in the bulk copies
            const int64_t blk = t * T + blt;
            const uint32_t rec_s = sbase + Lay::kOffRing + s * stage_bytes + blt * kRec;

            // W = sum_p q_p * (s_p / alpha_p) in shard order.  `scaled`: every
            // factor is formed 2^64 times larger (s_p 2^64 / alpha_p), and the
            // records are read again from global memory (the stage is gone).
            float w[LC];
            auto accumulate = [&](auto scaled) {
                constexpr bool kScaled = decltype(scaled)::value;
                auto factor = [&](uint2 meta) {
                    const float sv = kScaled ? __fmul_rn(__uint_as_float(meta.y), kTinyUp) : __uint_as_float(meta.y);
                    return __fdividef(sv, __uint_as_float(meta.x));
                };
#pragma unroll
                for (int k = 0; k < LC; k++)
                    w[k] = 0.f;
                // s_p / alpha_p below is within 2 ulp (alpha_p <= 1e15 is far from
                // the range where the fast quotient underflows).
                if (active && !from_global && !kScaled) {
                    const uint32_t r0 = rec_s + LC * part;
#pragma unroll(PFIX > 0 ? PFIX : 1)
                    for (int p = 0; p < P; p++) {
                        const uint32_t r = r0 + p * Lay::kRunBytes;
                        uint32_t words[LW];
#pragma unroll
                        for (int h = 0; h < LW / 2; h++) {
                            const uint2 a = lds64(r + 8 * h);
                            words[2 * h] = a.x;
                            words[2 * h + 1] = a.y;
                        }
                        accumulate_shard<CODE>(w, words, factor(lds64(r - LC * part + B)));
                    }
                } else if (active) {
                    // The tile's odd last record is not in the bulk copies (and
                    // the rare scaled pass reads every record again from there).
#pragma unroll 1
                    for (int p = 0; p < P; p++) {
                        const uint8_t *r = shard_ptr[p] + blk * kRec;
                        uint32_t words[LW];
#pragma unroll
                        for (int h = 0; h < LW / 2; h++) {
                            const uint2 a = ldg_u2(r + LC * part + 8 * h);
                            words[2 * h] = a.x;
                            words[2 * h + 1] = a.y;
                        }
                        accumulate_shard<CODE>(w, words, factor(ldg_u2(r + B)));
                    }
                }
            };
            accumulate(std::false_type{});
            if (sub == MUL - 1) {
                // The stage is read: hand it back to the loader.
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar(s));
            }

            // Energy |W|^2 and max|W| over the block's threads.
            float e = 0.f, wmax = 0.f;
            auto energy_max = [&]() {
                float2 e2 = make_float2(0.f, 0.f);
                wmax = 0.f;
#pragma unroll
                for (int k = 0; k < LC; k += 2) {
                    const float2 wi = make_float2(w[k], w[k + 1]);
                    e2 = fma2(wi, wi, e2);
                    wmax = max3(wmax, fabsf(w[k]), fabsf(w[k + 1]));
                }
                e = e2.x + e2.y;
#pragma unroll
                for (int d = 1; d < Lay::kLpb; d <<= 1) {
                    e = e + __shfl_xor_sync(kFullMask, e, d);
                    wmax = fmaxf(wmax, __shfl_xor_sync(kFullMask, wmax, d));
                }
            };
            energy_max();
            // A sum below 2^-80 (the near-zero region, where the factors
            // s_p / alpha_p are subnormal or zero in binary32, or an exact
            // cancellation) is summed again with scaled factors; its results
            // are scaled back by post = 2^-64 below.  DS only keeps the
            // unscaled sum, which is then the decoded shards' FP32 sum itself
            // (products q s_p, no rotation, alpha = 1).
            const bool tiny = active && !ds_only && wmax < kTinySum;
            if (__any_sync(kFullMask, tiny)) {     // warp-uniform, rare
                if (tiny)
                    accumulate(std::true_type{});
                energy_max();                       // the other blocks get the same values again
            }
            const float post = tiny ? kTinyDown : 1.0f;

            // post = 2^-64 where W was summed 2^64 times larger (1 elsewhere).
            const float m = __fmul_rn(__fmul_rn(e, post), post * (1.0f / B));
            const float alpha = adaptive ? __fdiv_rn(kTau, __fsqrt_rn(m + kEps)) : 1.0f;
            constexpr float qmax = CODE == 0 ? 448.0f : CODE == 1 ? 57344.0f : 127.0f;
            float sc = 0.f, kq = 0.f;
            if (!dual_scale) {          // ASH only: codes of alpha' W, s' = 1
                sc = 1.0f;
                kq = __fmul_rn(alpha, post);
            } else if (wmax > 0.f) {
                sc = __fdiv_rn(__fmul_rn(__fmul_rn(alpha, wmax), post), qmax);
                kq = __fdiv_rn(qmax, wmax);
            }
            uint32_t o[LW];
#pragma unroll
            for (int j = 0; j < LW; j++)
                o[j] = 0u;
            if (wmax > 0.f && !ds_only) {
#pragma unroll
                for (int j = 0; j < LW; j++)
                    o[j] = encode4_scaled(CODE, make_float2(w[4 * j], w[4 * j + 1]),
                                          make_float2(w[4 * j + 2], w[4 * j + 3]), kq);
            } else if (ds_only && sc >= kDivFastMin) {
                // DS only: W is the sum of the decoded shards itself (no
                // rotation, alpha = 1); its codes are W / s' correctly rounded.
                const float srcp = __frcp_rn(sc);
#pragma unroll
                for (int j = 0; j < LW; j++) {
                    const float2 u0 = div2_by(make_float2(w[4 * j], w[4 * j + 1]), sc, srcp);
                    const float2 u1 = div2_by(make_float2(w[4 * j + 2], w[4 * j + 3]), sc, srcp);
                    o[j] = encode4(CODE, u0.x, u0.y, u1.x, u1.y);
                }
            } else if (ds_only && wmax > 0.f) {
                // DS only with a tiny s': IEEE division.
#pragma unroll
                for (int j = 0; j < LW; j++)
                    o[j] = encode4(CODE, __fdiv_rn(w[4 * j], sc), __fdiv_rn(w[4 * j + 1], sc),
                                   __fdiv_rn(w[4 * j + 2], sc), __fdiv_rn(w[4 * j + 3], sc));
            }
            if (active) {
                uint8_t *rec = args.out + blk * kRec;
                // Records are 8-byte aligned: 8-byte stores.
#pragma unroll
                for (int h = 0; h < LW / 2; h++)
                    *reinterpret_cast<uint2 *>(rec + LC * part + 8 * h) = make_uint2(o[2 * h], o[2 * h + 1]);
                if (part == 0)
                    *reinterpret_cast<uint2 *>(rec + B) = make_uint2(__float_as_uint(alpha), __float_as_uint(sc));
            }
            }   // sub
        }
    }
}

template <int B, int CODE, int PFIX = 0>
KernelInfo info()
{
    using Lay = ReduceLayoutFor<B, PFIX>;
    return KernelInfo{reinterpret_cast<void *>(&taco_shard_reduce_kernel<B, CODE, PFIX>), Lay::kSmem, kRThreads,
                      Lay::kT, kRThreads / 32};
}

template <int CODE, int PFIX = 0>
KernelInfo info_for_block(int block)
{
    switch (block) {
    case 32: return info<32, CODE, PFIX>();
    case 64: return info<64, CODE, PFIX>();
    case 128: return info<128, CODE, PFIX>();
    case 256: return info<256, CODE, PFIX>();
    case 512: return info<512, CODE, PFIX>();
    default: return KernelInfo{};
    }
}

template <int PFIX>
KernelInfo info_for_code(int block, int code)
{
    switch (code) {
    case 0: return info_for_block<0, PFIX>(block);
    case 1: return info_for_block<1, PFIX>(block);
    case 2: return info_for_block<2, PFIX>(block);
    default: return KernelInfo{};
    }
}

}  // namespace

KernelInfo reduce_kernel_info(int block, int code, int num_shards)
{
    // The tensor-parallel degrees 2, 4, 8 and 16 (the owner reduces that many
    // segments) have kernels with the shard loop unrolled, for every code
    // format and block size: 2 and 4 with 32 codes per thread, 16 with a ring
    // of exactly three stages.  Other counts take a generic kernel: 1 and 3
    // the one with 32 codes per thread (16384 x 8192, 3 shards: 54.3 -> 33.2 us),
    // 5 to 15 the one with 16.
    if (TACO_REDUCE_FIXED_SHARDS) {
        switch (num_shards) {
        case 2: return info_for_code<2>(block, code);
        case 4: return info_for_code<4>(block, code);
        case 8: return info_for_code<8>(block, code);
        case 16: return info_for_code<16>(block, code);
        default: break;
        }
    }
    return num_shards <= 4 ? info_for_code<-4>(block, code) : info_for_code<0>(block, code);
}

cudaError_t launch_reduce(int block, int code, const ReduceArgs &args, uint32_t *fault, int grid, cudaStream_t stream)
{
    const KernelInfo ki = reduce_kernel_info(block, code, args.num_shards);
    if (!ki.fn)
        return cudaErrorInvalidValue;
    ReduceArgs a = args;
    void *params[] = {&a, &fault};
    return launch_kernel(ki.fn, grid, ki.threads, ki.smem, stream, params);
}

}  // namespace taco
