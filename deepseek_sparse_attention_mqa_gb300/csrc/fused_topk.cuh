// fused_topk.cuh -- the top-k phase of the fused indexer score + top-k kernels.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709), commit notes:
// the indexer is one op, indexer_score_topk, that scores the paged K cache and
// returns each row's top-k token positions.  Here a logits kernel that is asked
// for the top-k too runs this phase in every CTA once its own tiles are scored:
//  - each work unit's rows are selected by the ONE CTA that scored the unit's
//    last outstanding tiles: every CTA adds the number of the unit's tiles it
//    scored to the unit's counter (a caller workspace word), after a fence that
//    publishes its logits, and the CTA whose addition completes the count
//    selects the unit's rows (and puts the counter back to zero for the next
//    call) -- no CTA ever waits for another;
//  - the selection reads the logits just written, from L2, with a single-CTA
//    radix/bin select (select_cta.cuh) whose keys are cached in the shared
//    memory the scoring stages no longer need;
//  - units with no visible token (no tiles) are written as -1 rows by the CTAs
//    in turn.
// The separate top-k launch, its cluster barriers and its re-read of the logits
// from HBM disappear; what remains is the selection of the rows that complete
// last, at the end of the kernel.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "logits_common.cuh"
#include "select_cta.cuh"

namespace dsa {

constexpr int kDoneCap = 64;  // completed units selected per round

// Shared memory the phase needs besides its candidate store and key cache.
__host__ __device__ constexpr uint32_t fused_phase_fixed_bytes()
{
    return static_cast<uint32_t>((sizeof(SelectSmem) + 4 * (kDoneCap + 4) + 15) / 16 * 16);
}

// Smallest free shared memory the phase works with: the fixed part plus a
// candidate store of kSelCandCached entries.
__host__ __device__ constexpr uint32_t fused_phase_min_bytes()
{
    return fused_phase_fixed_bytes() + 8u * kSelCandCached;
}

struct FusedPhaseArgs {
    const SchedUnit* units;
    int num_units;
    int total_tiles;
    int t0, t1, R, u0;      // this CTA's tile range, super-tile size and first unit
    bool has_tiles;
    const float* logits;
    int64_t logits_stride;
    int logits_width;
    int next_n;
    int ratio;
    int row_begin;
    const int32_t* context_lens;
    int32_t* status;
    uint8_t* smem;          // free shared memory (16-byte aligned) ...
    uint32_t smem_bytes;    // ... of this size
};

// Select row `row` (absolute) of a unit whose logits are complete.
__device__ __forceinline__ void fused_select_row(const FusedPhaseArgs& a, const FusedTopk& f, const UnitInfo& ui,
                                                 int row, SelectSmem& sh, uint8_t* dyn, uint32_t dyn_bytes)
{
    const int i = row - ui.seq * a.next_n;
    const int vis = min(visible_entries(ui.ctx_len, a.next_n, i, a.ratio), a.logits_width);
    const int64_t rloc = row - a.row_begin;
    int32_t* out = f.idx + rloc * f.idx_stride;
    if (f.count && threadIdx.x == 0)
        f.count[rloc] = min(vis, f.k);
    if (vis <= f.k) {
        select_short_row_cta(vis, f.k, out);
        return;
    }
    select_row_cta(a.logits + rloc * a.logits_stride, vis, f.k, out, sh, dyn, dyn_bytes);
}

// Every thread of the CTA calls this after the scoring phase, with every logits
// store of the CTA issued and TMEM released.
static __device__ __noinline__ void fused_topk_phase(const FusedPhaseArgs& a, const FusedTopk& f)
{
    SelectSmem& sh = *reinterpret_cast<SelectSmem*>(a.smem);
    int* s_done = reinterpret_cast<int*>(a.smem + sizeof(SelectSmem));   // [kDoneCap] + n + more
    const uint32_t fixed = fused_phase_fixed_bytes();
    uint8_t* dyn = a.smem + fixed;                        // candidate store + key cache
    const uint32_t dyn_bytes = a.smem_bytes - fixed;
    const int tid = threadIdx.x;

    // units without tiles (no visible token in any of their rows): -1 rows
    for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
        const UnitInfo ui = unit_info(fetch_unit(a.units, u));
        if (ui.tile_end != ui.tile_begin)
            continue;
        for (int j = 0; j < ui.nrows; ++j) {
            const int64_t rloc = ui.first_row + j - a.row_begin;
            if (f.count && tid == 0)
                f.count[rloc] = 0;
            select_short_row_cta(0, f.k, f.idx + rloc * f.idx_stride);
        }
    }
    if (!a.has_tiles)
        return;

    // this CTA's logits stores are published before any counter moves
    __threadfence();
    __syncthreads();
    SuperWalk w;
    int cur = -1, mine = 0, cur_tiles = 0;
    if (tid == 0) {
        const WalkParams wp{a.context_lens, a.next_n, a.num_units};
        w.start(wp, a.units, a.total_tiles, a.t0, a.t1, a.R, a.u0);
    }
    for (;;) {
        if (tid == 0) {
            int n = 0;
            bool more = true;
            while (n < kDoneCap) {
                const bool valid = w.valid();
                const int u = valid ? w.w.u : -1;
                if (u != cur) {
                    if (cur >= 0) {
                        const int old = atomicAdd(f.counters + cur, mine);
                        if (old + mine == cur_tiles) {
                            f.counters[cur] = 0;       // every contribution is in: ready for the next call
                            s_done[n++] = cur;
                        }
                    }
                    cur = u;
                    mine = 0;
                    cur_tiles = valid ? w.w.ui.tile_end - w.w.ui.tile_begin : 0;
                }
                if (!valid) {
                    more = false;
                    break;
                }
                mine += w.nt;
                w.next();
            }
            __threadfence();                             // the other CTAs' logits of completed units
            s_done[kDoneCap] = n;
            s_done[kDoneCap + 1] = more ? 1 : 0;
        }
        __syncthreads();
        const int n = s_done[kDoneCap];
        const bool more = s_done[kDoneCap + 1] != 0;
        for (int d = 0; d < n; ++d) {
            const UnitInfo ui = unit_info(fetch_unit(a.units, s_done[d]));
            for (int j = 0; j < ui.nrows; ++j)
                fused_select_row(a, f, ui, ui.first_row + j, sh, dyn, dyn_bytes);
        }
        __syncthreads();
        if (!more)
            break;
    }
}

}  // namespace dsa
