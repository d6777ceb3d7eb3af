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
    int seq, first_row, nrows, tile_begin, tile_end, vis_max;
};

__device__ __forceinline__ UnitInfo load_unit(const WalkParams& p, const SchedUnit* units,
                                              int total_tiles, int u)
{
    UnitInfo ui;
    const SchedUnit su = units[u];
    ui.seq = su.seq;
    ui.first_row = su.first_row;
    ui.nrows = su.nrows;
    ui.tile_begin = su.tile_begin;
    ui.tile_end = (u + 1 < p.num_units) ? units[u + 1].tile_begin : total_tiles;
    const int L = max(0, p.context_lens[su.seq]);
    ui.vis_max = visible_len(L, p.next_n, su.first_row + su.nrows - 1 - su.seq * p.next_n);
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

// Walks this CTA's tiles [t0, t1) unit by unit; identical in every role.
struct TileWalk {
    const WalkParams* p;
    const SchedUnit* units;
    int total_tiles;
    int u;
    UnitInfo ui;
    __device__ __forceinline__ void start(const WalkParams& pp, const SchedUnit* us, int total, int t0)
    {
        start_at(pp, us, total, t0, find_unit(us, pp.num_units, t0));
    }
    // start from a unit found beforehand (find_unit / find_unit_warp of t0)
    __device__ __forceinline__ void start_at(const WalkParams& pp, const SchedUnit* us, int total, int t0, int u0)
    {
        p = &pp;
        units = us;
        total_tiles = total;
        u = u0;
        ui = load_unit(pp, us, total, u);
        while (t0 >= ui.tile_end && u + 1 < pp.num_units) {
            ++u;
            ui = load_unit(pp, us, total, u);
        }
    }
    // Advance to the unit that owns tile t; returns true if the unit changed.
    __device__ __forceinline__ bool seek(int t)
    {
        bool changed = false;
        while (t >= ui.tile_end && u + 1 < p->num_units) {
            ++u;
            ui = load_unit(*p, units, total_tiles, u);
            changed = true;
        }
        return changed;
    }
};

}  // namespace dsa
