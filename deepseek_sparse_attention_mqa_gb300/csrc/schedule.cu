// schedule.cu -- device-side indexer schedule builder.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709), commit notes:
// the decode indexer schedule is produced by a single kernel directly into a
// fixed-address CUDA-graph buffer (instead of ~50 small launches plus a copy),
// and the scoring kernel consumes it instead of building its own; it records
// absolute row ids, so every prefill chunk has its own schedule.
//
// Here one CTA turns the device-resident context lengths into the unit list
// (rows of one sequence that share an MMA N dimension) and the prefix of
// 128-token tiles over the units.  Everything that depends only on host-known
// values (unit boundaries) is recomputed on the device too, so the buffer is
// self-contained and valid for every graph replay.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"

namespace dsa {
namespace {

constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads)
build_schedule_kernel(const int32_t* __restrict__ context_lens, int batch, int next_n, int ratio, int G,
                      int row_begin, int row_end, int num_units, int32_t* __restrict__ sched,
                      int32_t* __restrict__ status)
{
    __shared__ int32_t warp_tot[kSchedThreads / 32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    SchedUnit* units = reinterpret_cast<SchedUnit*>(sched + kSchedHeaderWords);
    if (tid == 0)
        carry_s = 0;
    __syncthreads();

    for (int base = 0; base < num_units; base += kSchedThreads) {
        const int u = base + tid;
        int seq = 0, first_row = 0, nrows = 0, tiles = 0, vis = 0, ctx = 0;
        if (u < num_units) {
            unit_rows_of(u, next_n, G, row_begin, row_end, &seq, &first_row, &nrows);
            if (seq < batch && nrows > 0) {
                const int L = context_lens[seq];
                ctx = L < 0 ? 0 : L;
                const int last_i = first_row + nrows - 1 - seq * next_n;
                vis = visible_entries(ctx, next_n, last_i, ratio);
                tiles = (vis + kTileTokens - 1) / kTileTokens;
            } else if (status) {
                atomicOr(status, DSA_DEV_SCHEDULE);
            }
        }
        // block-wide exclusive scan of tiles
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        if (lane == 31)
            warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o)
                    t += v;
            }
            warp_tot[lane] = t;   // inclusive over warps
        }
        __syncthreads();
        const int carry = carry_s;
        const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - tiles;
        if (u < num_units) {
            SchedUnit su;
            su.first_row = first_row;
            su.nrows = nrows;
            su.seq = seq;
            su.tile_begin = excl;
            su.tile_end = excl + tiles;
            su.vis_max = vis;
            su.ctx_len = ctx;
            su.pad = 0;
            units[u] = su;
        }
        __syncthreads();
        if (tid == 0)
            carry_s = carry + warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) {
        sched[0] = kSchedMagic;
        sched[1] = num_units;
        sched[2] = G;
        sched[3] = row_begin;
        sched[4] = row_end;
        sched[5] = next_n;
        sched[6] = carry_s;
        sched[7] = ratio;
    }
}

}  // namespace

dsa_status launch_build_schedule(const int32_t* context_lens, int batch, int next_n, int ratio,
                                 int rows_per_unit, int row_begin, int row_end, int num_units,
                                 int32_t* sched, int32_t* status, cudaStream_t stream)
{
    build_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(context_lens, batch, next_n, ratio,
                                                           rows_per_unit, row_begin, row_end,
                                                           num_units, sched, status);
    return check_launch();
}

}  // namespace dsa
