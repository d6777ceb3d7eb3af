// logits_common.cuh -- schedule walking shared by the indexer logits kernels.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dsa {

// Fields of the logits launch every role needs to walk the schedule.
struct WalkParams {
    const int32_t* context_lens;
    int next_n;
    int num_units;
};

struct UnitInfo {
    int seq, first_row, nrows, tile_begin, tile_end, vis_max, ctx_len;
};

// One schedule record (32 bytes, two 16-byte loads).
__device__ __forceinline__ SchedUnit fetch_unit(const SchedUnit* units, int u)
{
    const int4* src = reinterpret_cast<const int4*>(units + u);
    const int4 a = src[0], b = src[1];
    SchedUnit su;
    su.first_row = a.x;
    su.nrows = a.y;
    su.seq = a.z;
    su.tile_begin = a.w;
    su.tile_end = b.x;
    su.vis_max = b.y;
    su.ctx_len = b.z;
    su.pad = b.w;
    return su;
}

__device__ __forceinline__ UnitInfo unit_info(const SchedUnit& su)
{
    UnitInfo ui;
    ui.seq = su.seq;
    ui.first_row = su.first_row;
    ui.nrows = su.nrows;
    ui.tile_begin = su.tile_begin;
    ui.tile_end = su.tile_end;
    ui.vis_max = su.vis_max;
    ui.ctx_len = su.ctx_len;
    return ui;
}

// Last unit whose tile_begin <= t (units with no tiles are skipped naturally).
__device__ __forceinline__ int find_unit(const SchedUnit* units, int num_units, int t)
{
    int lo = 0, hi = num_units - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (units[mid].tile_begin <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// find_unit by one whole warp: each round probes 32 evenly spaced units at
// once (one global-memory latency per round instead of one per halving), so a
// CTA finds its first unit in two rounds for up to 1024 units.  All 32 lanes
// must call it; every lane returns the same unit.
__device__ __forceinline__ int find_unit_warp(const SchedUnit* units, int num_units, int t)
{
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = num_units;                  // answer in [lo, hi); units[lo].tile_begin <= t
    while (hi - lo > 1) {
        const int span = hi - lo;
        const int idx = lo + static_cast<int>((static_cast<long long>(span) * lane) / 32);
        const unsigned le = __ballot_sync(0xffffffffu, units[idx].tile_begin <= t);
        const int k = 31 - __clz(le);            // last probe at or before t (lane 0 always is)
        const int nlo = lo + static_cast<int>((static_cast<long long>(span) * k) / 32);
        hi = k == 31 ? hi : lo + static_cast<int>((static_cast<long long>(span) * (k + 1)) / 32);
        lo = nlo;
    }
    return lo;
}

// Walks this CTA's tiles [t0, t1) unit by unit; identical in every role.  The
// record of the next unit is fetched as soon as a unit is entered, so a unit
// change costs no global-memory round trip.
struct TileWalk {
    const SchedUnit* units;
    int num_units;
    int u;
    UnitInfo ui;
    SchedUnit nx;            // record of unit u + 1 (when it exists)
    __device__ __forceinline__ void start(const WalkParams& pp, const SchedUnit* us, int total, int t0)
    {
        start_at(pp, us, total, t0, find_unit(us, pp.num_units, t0));
    }
    // start from a unit found beforehand (find_unit / find_unit_warp of t0)
    __device__ __forceinline__ void start_at(const WalkParams& pp, const SchedUnit* us, int, int t0, int u0)
    {
        units = us;
        num_units = pp.num_units;
        u = u0;
        ui = unit_info(fetch_unit(us, u));
        if (u + 1 < num_units)
            nx = fetch_unit(us, u + 1);
        while (t0 >= ui.tile_end && u + 1 < num_units)
            advance();
    }
    __device__ __forceinline__ void advance()
    {
        ++u;
        ui = unit_info(nx);
        if (u + 1 < num_units)
            nx = fetch_unit(units, u + 1);
    }
    // Advance to the unit that owns tile t; returns true if the unit changed.
    __device__ __forceinline__ bool seek(int t)
    {
        bool changed = false;
        while (t >= ui.tile_end && u + 1 < num_units) {
            advance();
            changed = true;
        }
        return changed;
    }
};

// Walks this CTA's super-tiles.  A super-tile is up to R consecutive 128-token
// tiles of ONE unit, aligned to the unit's first tile; it belongs to the CTA
// whose tile range [t0, t1) holds its first tile (it may run past t1).  Every
// role walks the same sequence, so the super-tile ordinal j is the same in all.
struct SuperWalk {
    TileWalk w;
    int R, t1, ts, nt;   // current super-tile: tiles [ts, ts + nt) of unit w.u

    __device__ __forceinline__ void settle()
    {
        if (ts >= w.ui.tile_end)
            ts = w.ui.tile_end;              // the next unit's first tile
        w.seek(ts);
        nt = min(R, w.ui.tile_end - ts);
    }
    __device__ __forceinline__ void start(const WalkParams& wp, const SchedUnit* units, int total, int t0,
                                          int t1_, int R_, int u0)
    {
        R = R_;
        t1 = t1_;
        w.start_at(wp, units, total, t0, u0);
        const int off = max(0, t0 - w.ui.tile_begin);
        ts = w.ui.tile_begin + ((off + R - 1) / R) * R;
        settle();
    }
    __device__ __forceinline__ bool valid() const { return ts < t1 && nt > 0; }
    __device__ __forceinline__ void next()
    {
        ts += R;
        settle();
    }
    // first tile of the super-tile inside its unit
    __device__ __forceinline__ int tile_in_unit() const { return ts - w.ui.tile_begin; }
};

// ------------------------------------------------------------ inline schedule
//
// A logits launch without a schedule buffer builds the unit records itself, in
// shared memory, when there are at most kInlineUnits units (a decode batch of up
// to 256 sequences): every CTA computes the same records from the context
// lengths in its prologue, which costs about what reading a prebuilt schedule
// costs and saves the schedule kernel's launch.  ("Add fp4 indexer for dsv4",
// commit notes: with a prebuilt schedule buffer the scoring kernel skips its own
// build.)  kInlineUnits is in common.cuh.
constexpr uint32_t kInlineScratchBytes = 160;   // 33 ints of scan scratch, 16-byte multiple

// All threads of the CTA call this (blockDim.x >= num_units, blockDim.x <= 1024).
// Writes records [0, num_units) to `su` exactly as the schedule kernel does and
// returns the total number of 128-token tiles.
__device__ __forceinline__ int build_inline_units(SchedUnit* su, int* scratch, const int32_t* context_lens,
                                                  int batch, int next_n, int ratio, int G, int row_begin,
                                                  int row_end, int num_units, int32_t* status)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = static_cast<int>(blockDim.x + 31) >> 5;
    int seq = 0, first_row = 0, nrows = 0, tiles = 0, vis = 0, ctx = 0;
    if (tid < num_units) {
        unit_rows_of(tid, next_n, G, row_begin, row_end, &seq, &first_row, &nrows);
        if (seq < batch && nrows > 0) {
            const int L = context_lens[seq];
            ctx = L < 0 ? 0 : L;
            vis = visible_entries(ctx, next_n, first_row + nrows - 1 - seq * next_n, ratio);
            tiles = (vis + kTileTokens - 1) / kTileTokens;
        } else if (status) {
            atomicOr(status, DSA_DEV_SCHEDULE);
        }
    }
    // block-wide exclusive scan of the tile counts
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += v;
        }
        scratch[lane] = t;                     // inclusive over warps
    }
    __syncthreads();
    const int excl = (warp > 0 ? scratch[warp - 1] : 0) + incl - tiles;
    if (tid < num_units) {
        SchedUnit r;
        r.first_row = first_row;
        r.nrows = nrows;
        r.seq = seq;
        r.tile_begin = excl;
        r.tile_end = excl + tiles;
        r.vis_max = vis;
        r.ctx_len = ctx;
        r.pad = 0;
        su[tid] = r;
    }
    const int total = scratch[nw - 1];
    __syncthreads();
    return total;
}

}  // namespace dsa
