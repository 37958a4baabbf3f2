// taco_sched.cuh -- dynamic tile scheduling for the persistent-style kernels
// (compress, decompress, shard reduce) with cluster launch control.
//
// The grid has one CTA per tile, and shared memory admits one CTA per SM.  A
// running CTA takes its own tile (item 0), then asks the hardware to cancel
// CTAs that have not started yet and takes their tiles (items 1, 2, ...), so
// SMs that get more memory bandwidth take more tiles and all finish together.
//
// Only the producer thread (the one that issues the tile loads) issues and
// reads cancel requests: it keeps kSchedAhead of them in flight, reads the
// responses in order and stops requesting at the first failed one, so the CTA
// never requests again after it has seen a failure.  It hands every item's
// tile to the other roles through a ring of kTileRing shared-memory slots,
// each with an mbarrier (one arrival per publication), and publishes an item
// only when it issues that item's loads: by then the stage the item will use
// has been released by the item before it, so no reader can mistake an older
// phase of a stage barrier for the item's.  After the last tile it publishes
// -1 for `groups` items, one for each role that takes every groups-th item.
#pragma once

#include <cstdint>

#include "taco_device.cuh"
#include "taco_tcgen05.cuh"

namespace taco {

constexpr int kSchedSlots = 16;   // cancel-response slots
#ifndef TACO_SCHED_AHEAD
#define TACO_SCHED_AHEAD 1
#endif
// Cancel requests in flight.  One is enough to hide the round trip behind a
// tile's loads; with more, the CTAs that ask first claim most of the tiles of
// a small grid before the others have asked once (0.2-0.4 us slower per
// launch at 33.5 M elements).
constexpr int kSchedAhead = TACO_SCHED_AHEAD;
constexpr int kTileRing = 16;     // published-tile slots
#ifndef TACO_L2_PREFETCH_COMPRESS
#define TACO_L2_PREFETCH_COMPRESS 3
#endif
#ifndef TACO_L2_PREFETCH_DECOMPRESS
#define TACO_L2_PREFETCH_DECOMPRESS 2
#endif
#ifndef TACO_L2_PREFETCH_REDUCE
#define TACO_L2_PREFETCH_REDUCE 2
#endif
// Tiles whose input a CTA prefetches into L2 before its dependency wait, per
// kernel: its own, then (a guess at what it or its neighbours take next) those
// one, two, ... SM counts further on.
constexpr int kL2PrefetchCompress = TACO_L2_PREFETCH_COMPRESS;
constexpr int kL2PrefetchDecompress = TACO_L2_PREFETCH_DECOMPRESS;
constexpr int kL2PrefetchReduce = TACO_L2_PREFETCH_REDUCE;

// Shared-memory bytes: responses (16 B each, 16-byte aligned first), tiles
// (8 B each) and the two sets of mbarriers.
constexpr int kSchedBytes = 16 * kSchedSlots + 8 * kTileRing + 8 * kSchedSlots + 8 * kTileRing;

struct TileSched {
    uint32_t base;       // shared-memory address of the area (16-byte aligned)
    uint32_t *fault;
    uint32_t fault_bit;

    __device__ uint32_t resp(int q) const { return base + 16u * q; }
    __device__ uint32_t tile_addr(int r) const { return base + 16u * kSchedSlots + 8u * r; }
    __device__ uint32_t resp_bar(int q) const { return base + 16u * kSchedSlots + 8u * kTileRing + 8u * q; }
    __device__ uint32_t tile_bar(int r) const
    {
        return base + 16u * kSchedSlots + 8u * kTileRing + 8u * kSchedSlots + 8u * r;
    }

    // One thread, before the CTA's first barrier (followed by fence_mbar_init).
    __device__ void init() const
    {
        for (int q = 0; q < kSchedSlots; q++)
            mbar_init(resp_bar(q), 1);
        for (int r = 0; r < kTileRing; r++)
            mbar_init(tile_bar(r), 1);
    }

    // ---- producer thread ----------------------------------------------------

    // Cancel request j >= 1 (answers item j).
    __device__ void request(int j) const
    {
        const int q = (j - 1) % kSchedSlots;
        mbar_arrive_expect_tx(resp_bar(q), 16);
        clc_try_cancel(resp(q), resp_bar(q));
    }

    // Tile of item j >= 1 from its response, or -1 if the request failed (or
    // the wait timed out, which also sets the fault bit).
    __device__ int64_t response(int j) const
    {
        const int q = (j - 1) % kSchedSlots;
        if (!mbar_wait_bounded_thread(resp_bar(q), ((j - 1) / kSchedSlots) & 1, fault, fault_bit))
            return -1;
        const int64_t t = clc_response_ctaid_x(resp(q));
        if (t >= static_cast<int64_t>(gridDim.x)) {   // not a tile of this grid: give up, flag it
            atomicOr(fault, fault_bit);
            return -1;
        }
        return t;
    }

    // Waits for the responses of requests from .. to (issued, not read), so
    // that none is still being written when the CTA exits.
    __device__ void drain(int from, int to) const
    {
        for (int j = from; j <= to; j++)
            mbar_wait_bounded_thread(resp_bar((j - 1) % kSchedSlots), ((j - 1) / kSchedSlots) & 1, fault,
                                     fault_bit);
    }

    __device__ void publish(int i, int64_t tile) const
    {
        const int r = i % kTileRing;
        asm volatile("st.shared.s64 [%0], %1;" ::"r"(tile_addr(r)), "l"(tile) : "memory");
        mbar_arrive(tile_bar(r));   // release: the store is visible to whoever waits
    }

    // Publishes -1 for items i .. i + groups - 1.
    __device__ void publish_end(int i, int groups) const
    {
        for (int k = 0; k < groups; k++)
            publish(i + k, -1);
    }

    // ---- readers ------------------------------------------------------------

    __device__ int64_t read_tile(int i) const
    {
        int64_t t;
        asm volatile("ld.shared.s64 %0, [%1];" : "=l"(t) : "r"(tile_addr(i % kTileRing)) : "memory");
        return t;
    }

    // Tile of item i, or -1 at the end (whole warp; the outcome is uniform).
    __device__ int64_t tile_warp(int i) const
    {
        if (!mbar_wait_bounded(tile_bar(i % kTileRing), (i / kTileRing) & 1, fault, fault_bit))
            return -1;
        return read_tile(i);
    }

    // Same for a single thread.
    __device__ int64_t tile_thread(int i) const
    {
        if (!mbar_wait_bounded_thread(tile_bar(i % kTileRing), (i / kTileRing) & 1, fault, fault_bit))
            return -1;
        return read_tile(i);
    }
};

}  // namespace taco
