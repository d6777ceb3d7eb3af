// logits_fp8.cu -- paged lightning-indexer MQA logits over an FP8 (e4m3) K cache.
//
//   logits[r][s] = k_scale[s] * sum_h w[r][h] * relu(q[r][h] . k[s])
//
// Prior art on the pages ("SM120 FP8 paged MQA page 32", vllm-project/DeepGEMM #14,
// Summary and review): one TMA copy per physical page, never a tile that
// straddles two non-contiguous pages (BLOCK_KV = min(PAGE_KV, 64)), several
// TMA warps each owning a KV group, 2-3 stages to fit SM120's 99 KiB.
//
// GB300 design (one persistent CTA per SM, warp-specialised):
//   warps 0,10-12  TMA producers, taking tiles round-robin: per 128-token tile,
//               one 3-D box per physical page (2 boxes at page 64, 4 at page 32)
//               into a 128B/64B/32B-swizzled K-major stage, plus one box of
//               per-token fp32 scales per page; warp 0 also loads the unit's q
//               rows ([rows x heads, D], K-major) once per unit.  A single
//               producer warp spends about twice the HBM time of a tile on the
//               copies' issue and the page bookkeeping, so several share it.
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer, kind::f8f6f4:
//               D[128 tokens x N] += K_tile[128 x D] * Q[N x D]^T, N = rows x heads.
//               Each TMEM lane is one token and each column one (row, head).
//   warps 2-9   epilogue, two warpgroups taking alternate tiles (so two warps per
//               scheduler hide each other's TMEM-load and barrier latency):
//               tcgen05.ld of the thread's own lane, then the whole relu /
//               head-weighting / k_scale reduction is thread-local (no shuffles),
//               and each warp stores 32 consecutive logits per row.
//   Four TMEM accumulators let the epilogues of earlier tiles overlap the MMA of
//   later ones; the stage ring keeps enough K bytes in flight to cover HBM latency.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "host.h"
#include "logits_common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kMaxStages = 16;
constexpr int kEpiWarps = 8;
constexpr int kProd = 4;        // TMA producer warps (warp 0 and the warps after the epilogue)
constexpr int kThreads = 32 * (2 + kEpiWarps + kProd - 1);  // producers, MMA, two epilogue warpgroups
constexpr int kPageCache = 512; // physical page ids cached by each producer warp
constexpr int kMaxAcc = 4;      // TMEM accumulators in flight

struct LogitsParams {
    const int32_t* sched;
    const int32_t* context_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    int max_pages;
    int num_pages;
    int page_kv;
    int next_n;
    int row_begin;
    int row_end;
    int num_units;
    int rows_per_unit;
    const float* weights;
    float* logits;
    int64_t logits_stride;
    int logits_width;
    int32_t* status;
    int stages;
    int n_cols;         // MMA N (multiple of 16)
    uint32_t acc_cols;  // TMEM columns per accumulator (power of two >= 32, >= n_cols)
    int n_acc;          // accumulators (n_acc * acc_cols <= 512, power of two total)
    uint32_t q_buf_bytes;
};

template <int D>
struct Fp8Tile {
    static constexpr uint32_t kTileBytes = kTileTokens * D;   // K bytes per stage
    static constexpr uint32_t kLayout = D == 128 ? kLayoutSw128 : (D == 64 ? kLayoutSw64 : kLayoutSw32);
    static constexpr uint32_t kSbo = 8 * D;                    // 8 rows per swizzle atom
    static constexpr int kKSteps = D / 32;                      // K = 32 bytes per MMA
};

// Shared memory map (offsets from a 1024-aligned base).
struct SmemMap {
    uint32_t k_off, q_off, sc_off, w_off, pc_off, bar_off, misc_off, total;
};

__host__ __device__ __forceinline__ SmemMap smem_map(int D, int stages, uint32_t q_buf_bytes)
{
    SmemMap m;
    m.k_off = 0;
    m.q_off = m.k_off + stages * kTileTokens * D;
    m.sc_off = m.q_off + 2 * q_buf_bytes;
    m.w_off = m.sc_off + stages * kTileTokens * 4;
    m.pc_off = m.w_off + kEpiWarps * kMaxUnitCols * 4;       // one weight copy per epilogue warp
    m.bar_off = m.pc_off + kProd * kPageCache * 4;
    m.misc_off = m.bar_off + (2 * kMaxStages + 2 * kMaxAcc + 4 + 1) * 8;
    m.total = m.misc_off + 16;
    return m;
}

template <int D, int H>
__global__ void __launch_bounds__(kThreads, 1)
logits_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_q, const LogitsParams p)
{
    using T = Fp8Tile<D>;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemMap mp = smem_map(D, p.stages, p.q_buf_bytes);
    uint8_t* sK = smem + mp.k_off;
    uint8_t* sQ = smem + mp.q_off;
    float* sS = reinterpret_cast<float*>(smem + mp.sc_off);
    float* sW = reinterpret_cast<float*>(smem + mp.w_off);
    int* s_pages = reinterpret_cast<int*>(smem + mp.pc_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + mp.bar_off);
    uint64_t* full_bar = bars;                       // [stages]
    uint64_t* empty_bar = bars + kMaxStages;         // [stages]
    uint64_t* accf_bar = bars + 2 * kMaxStages;      // [kMaxAcc]
    uint64_t* acce_bar = accf_bar + kMaxAcc;         // [kMaxAcc]
    uint64_t* qf_bar = acce_bar + kMaxAcc;           // [2]
    uint64_t* qe_bar = qf_bar + 2;                   // [2]
    uint64_t* done_bar = qe_bar + 2;                 // [1]
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(smem + mp.misc_off);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + mp.misc_off + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- schedule header (uniform over the CTA, checked before any allocation)
    const int32_t* hdr = p.sched;
    const SchedUnit* units = reinterpret_cast<const SchedUnit*>(p.sched + kSchedHeaderWords);
    if (hdr[0] != kSchedMagic || hdr[1] != p.num_units || hdr[2] != p.rows_per_unit ||
        hdr[3] != p.row_begin || hdr[4] != p.row_end || hdr[5] != p.next_n) {
        if (threadIdx.x == 0 && p.status)
            atomicOr(p.status, DSA_DEV_SCHEDULE);
        return;
    }
    const int total_tiles = hdr[6];
    const int t0 = static_cast<int>((static_cast<long long>(blockIdx.x) * total_tiles) / gridDim.x);
    const int t1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * total_tiles) / gridDim.x);
    if (t0 >= t1 || p.num_units == 0)
        return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1 + 4);   // MMA commit + the tile's 4 epilogue warps
        }
        for (int a = 0; a < kMaxAcc; ++a) {
            mbar_init(smem_u32(&accf_bar[a]), 1);
            mbar_init(smem_u32(&acce_bar[a]), 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&qf_bar[a]), 1);
            mbar_init(smem_u32(&qe_bar[a]), 1);
        }
        mbar_init(smem_u32(done_bar), 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_s);
        tma_prefetch_map(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), p.n_acc * p.acc_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const WalkParams wp{p.context_lens, p.next_n, p.num_units};
    const int P = p.page_kv;
    const int pages_per_tile = kTileTokens / P;

    if (warp == 0 || warp >= 2 + kEpiWarps) {
        // =========================== TMA producers ==========================
        // kProd warps share the tile stream: producer pi issues the tiles whose
        // CTA-local ordinal j has j % kProd == pi, so the per-tile work around
        // the copies (page lookup, barrier waits, descriptor fetch) of several
        // tiles overlaps.  The stage count is a multiple of kProd, so every
        // stage has exactly one producer and its empty/full phases advance in
        // that producer's order.  Producer 0 also loads each unit's q rows.
        // Physical page ids are fetched by all 32 lanes at once into the warp's
        // own shared-memory cache (one global-memory latency per refill).
        const int pi = warp == 0 ? 0 : warp - (1 + kEpiWarps);
        int* my_pages = s_pages + pi * kPageCache;
        TileWalk w;
        w.start(wp, units, total_tiles, t0);
        int ucount = 0;
        long long issued = 0;
        int pc_unit = -1, pc_lp0 = 0, pc_cnt = 0;
        for (int t = t0; t < t1; ++t) {
            if (__any_sync(0xffffffffu, *s_abort))
                break;
            const bool changed = w.seek(t) || (t == t0);
            int ok = 1;
            if (changed) {
                if (pi == 0 && lane == 0) {
                    const int qb = ucount & 1;
                    ok = mbar_wait(smem_u32(&qe_bar[qb]), ((ucount >> 1) & 1) ^ 1);
                    if (ok) {
                        mbar_arrive_expect_tx(smem_u32(&qf_bar[qb]), static_cast<uint32_t>(p.n_cols) * D);
                        tma_load_2d(smem_u32(sQ + qb * p.q_buf_bytes), &tm_q, smem_u32(&qf_bar[qb]), 0,
                                    w.ui.first_row * H);
                    }
                }
                ++ucount;
            }
            const int j = t - t0;
            if (j % kProd != pi) {
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0)
                        *s_abort = 1;
                    break;
                }
                continue;
            }
            const int stage = j % p.stages;
            const uint32_t phase = static_cast<uint32_t>((j / p.stages) & 1);
            const int tt = t - w.ui.tile_begin;              // tile index inside the unit
            const int lp_first = tt * pages_per_tile;
            if (w.u != pc_unit || lp_first + pages_per_tile > pc_lp0 + pc_cnt) {
                // refill: this unit's pages from lp_first up to what this CTA will use
                const int tiles_here = min(t1, w.ui.tile_end) - w.ui.tile_begin;
                const int lp_vis = (w.ui.vis_max + P - 1) / P;
                const int lp_end = min(tiles_here * pages_per_tile, lp_vis);
                const int cnt = min(kPageCache, max(lp_end - lp_first, pages_per_tile));
                __syncwarp();
                for (int i = lane; i < cnt; i += 32) {
                    const int lp = lp_first + i;
                    int pg = -1;
                    if (lp < lp_vis && lp < p.max_pages)
                        pg = p.block_table[static_cast<int64_t>(w.ui.seq) * p.bt_stride + lp];
                    my_pages[i] = pg;
                }
                __syncwarp();
                pc_unit = w.u;
                pc_lp0 = lp_first;
                pc_cnt = cnt;
            }
            if (lane == 0 && ok) {
                ok = mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1);
                if (ok) {
                    int phys[kTileTokens / 32];
                    uint32_t bytes = 0;
                    for (int jp = 0; jp < pages_per_tile; ++jp) {
                        const int lp = lp_first + jp;
                        phys[jp] = -1;
                        if (lp * P < w.ui.vis_max) {
                            const int pg = my_pages[lp - pc_lp0];
                            if (pg >= 0 && pg < p.num_pages) {
                                phys[jp] = pg;
                                bytes += static_cast<uint32_t>(P) * (D + 4);
                            } else if (p.status) {
                                atomicOr(p.status, DSA_DEV_BAD_PAGE);
                            }
                        }
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    for (int jp = 0; jp < pages_per_tile; ++jp) {
                        if (phys[jp] < 0)
                            continue;
                        tma_load_3d(smem_u32(sK + stage * T::kTileBytes + jp * P * D), &tm_k, fb, 0, 0, phys[jp]);
                        tma_load_2d(smem_u32(sS + stage * kTileTokens + jp * P), &tm_s, fb, 0, phys[jp]);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0)
                    *s_abort = 1;
                break;
            }
            ++issued;
        }
        // drain: every copy this warp issued has landed before the CTA exits
        // (its stages are its own, so the last stages/kProd of its tiles are
        // the only ones whose full phase may still be pending)
        if (lane == 0) {
            const long long per = p.stages / kProd;
            const long long lo = issued > per ? issued - per : 0;
            for (long long n = lo; n < issued; ++n) {
                const long long jj = pi + n * kProd;
                mbar_wait(smem_u32(&full_bar[jj % p.stages]), static_cast<uint32_t>((jj / p.stages) & 1));
            }
            if (pi == 0)
                for (int u = ucount > 2 ? ucount - 2 : 0; u < ucount; ++u)
                    mbar_wait(smem_u32(&qf_bar[u & 1]), static_cast<uint32_t>((u >> 1) & 1));
        }
    } else if (warp == 1) {
        // =========================== MMA issuer =============================
        if (lane == 0) {
            const uint32_t idesc = make_idesc(0, 0, 0, 128, static_cast<uint32_t>(p.n_cols));
            TileWalk w;
            w.start(wp, units, total_tiles, t0);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            int ucount = 0, qb = 0;
            for (int t = t0; t < t1 && !*s_abort; ++t) {
                const bool changed = w.seek(t) || (t == t0);
                if (changed) {
                    qb = ucount & 1;
                    if (!mbar_wait(smem_u32(&qf_bar[qb]), (ucount >> 1) & 1)) {
                        *s_abort = 1;
                        break;
                    }
                    ++ucount;
                }
                if (!mbar_wait(smem_u32(&acce_bar[acc]), acc_phase ^ 1) ||
                    !mbar_wait(smem_u32(&full_bar[stage]), phase)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * p.acc_cols;
                const uint32_t a_base = smem_u32(sK + stage * T::kTileBytes);
                const uint32_t b_base = smem_u32(sQ + qb * p.q_buf_bytes);
#pragma unroll
                for (int k = 0; k < T::kKSteps; ++k) {
                    const uint64_t ad = make_smem_desc(a_base + k * 32, 16, T::kSbo, T::kLayout);
                    const uint64_t bd = make_smem_desc(b_base + k * 32, 16, T::kSbo, T::kLayout);
                    umma_f8f6f4(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
                }
                umma_commit(smem_u32(&empty_bar[stage]));
                umma_commit(smem_u32(&accf_bar[acc]));
                const bool unit_ends = (t + 1 == t1) || (t + 1 >= w.ui.tile_end);
                if (unit_ends)
                    umma_commit(smem_u32(&qe_bar[qb]));
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++acc == p.n_acc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(smem_u32(done_bar));
            mbar_wait(smem_u32(done_bar), 0);
        }
    } else {
        // =========================== epilogue ===============================
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const int group = (warp - 2) >> 2;            // epilogue warpgroup: takes tiles t0+group, t0+group+2, ...
        const int tok = quarter * 32 + lane;          // token of this thread within the tile
        float* wS = sW + (warp - 2) * kMaxUnitCols;   // this warp's copy of the unit weights
        TileWalk w;
        w.start(wp, units, total_tiles, t0);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        int nchunks = 0, L = 0, i0 = 0;
        for (int t = t0; t < t1 && !__any_sync(0xffffffffu, *s_abort); ++t) {
            const bool changed = w.seek(t) || (t == t0);
            if (changed) {
                __syncwarp();
                const int ncols_valid = w.ui.nrows * H;
                nchunks = (ncols_valid + 31) / 32;
                const float* wsrc = p.weights + static_cast<int64_t>(w.ui.first_row) * H;
                for (int c = lane; c < kMaxUnitCols; c += 32)
                    wS[c] = c < ncols_valid ? wsrc[c] : 0.f;
                __syncwarp();
                L = max(0, p.context_lens[w.ui.seq]);
                i0 = w.ui.first_row - w.ui.seq * p.next_n;
                if (lane == 0 && group == 0 && p.status &&
                    visible_len(L, p.next_n, i0 + w.ui.nrows - 1) > p.logits_width)
                    atomicOr(p.status, DSA_DEV_WIDTH);
            }
            if (((t - t0) & 1) != group) {            // the other warpgroup's tile
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++acc == p.n_acc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
                continue;
            }
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[stage]), phase) &&
                                             mbar_wait(smem_u32(&accf_bar[acc]), acc_phase))) {
                *s_abort = 1;
                break;
            }
            tc_fence_after_sync();
            const float kscale = sS[stage * kTileTokens + tok];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&empty_bar[stage]));

            const int s = (t - w.ui.tile_begin) * kTileTokens + tok;
            const uint32_t t_acc = tmem_base + static_cast<uint32_t>(acc) * p.acc_cols +
                                   (static_cast<uint32_t>(quarter * 32) << 16);
            // store one finished logit of unit row i
            auto emit = [&](int i, float v) {
                if (i < w.ui.nrows) {
                    const int vis = min(visible_len(L, p.next_n, i0 + i), p.logits_width);
                    if (s < vis)
                        p.logits[static_cast<int64_t>(w.ui.first_row + i - p.row_begin) * p.logits_stride + s] =
                            kscale * v;
                }
            };
            float cur = 0.f;                           // running row sum (H >= 32)
            auto process = [&](const uint32_t (&r)[32], int c) {
                const float4* w4 = reinterpret_cast<const float4*>(wS + c * 32);
                if constexpr (H >= 32) {
                    // one row per chunk: 8 independent partial sums
                    float part[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        part[j] = 0.f;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 wv = w4[q4];
                        part[(4 * q4 + 0) & 7] = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * q4 + 0]), 0.f), part[(4 * q4 + 0) & 7]);
                        part[(4 * q4 + 1) & 7] = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * q4 + 1]), 0.f), part[(4 * q4 + 1) & 7]);
                        part[(4 * q4 + 2) & 7] = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * q4 + 2]), 0.f), part[(4 * q4 + 2) & 7]);
                        part[(4 * q4 + 3) & 7] = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * q4 + 3]), 0.f), part[(4 * q4 + 3) & 7]);
                    }
                    cur += ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
                    if (((c + 1) * 32) % H == 0) {
                        emit((c * 32) / H, cur);
                        cur = 0.f;
                    }
                } else {
                    // 32 / H rows per chunk, each summed over its H columns
                    constexpr int kRowsPerChunk = 32 / H;
                    float rs[kRowsPerChunk];
#pragma unroll
                    for (int i = 0; i < kRowsPerChunk; ++i)
                        rs[i] = 0.f;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 wv = w4[q4];
                        rs[(4 * q4 + 0) / H] = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * q4 + 0]), 0.f), rs[(4 * q4 + 0) / H]);
                        rs[(4 * q4 + 1) / H] = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * q4 + 1]), 0.f), rs[(4 * q4 + 1) / H]);
                        rs[(4 * q4 + 2) / H] = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * q4 + 2]), 0.f), rs[(4 * q4 + 2) / H]);
                        rs[(4 * q4 + 3) / H] = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * q4 + 3]), 0.f), rs[(4 * q4 + 3) / H]);
                    }
#pragma unroll
                    for (int i = 0; i < kRowsPerChunk; ++i)
                        emit(c * kRowsPerChunk + i, rs[i]);
                }
            };
            for (int c = 0; c < nchunks; c += 2) {
                uint32_t ra[32], rb[32];
                tmem_ld_32x32b_x32(t_acc + c * 32, ra);
                if (c + 1 < nchunks)
                    tmem_ld_32x32b_x32(t_acc + (c + 1) * 32, rb);
                tmem_ld_wait();
                if (c + 2 >= nchunks) {
                    // last TMEM reads of this accumulator are in registers: release it early
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&acce_bar[acc]));
                }
                process(ra, c);
                if (c + 1 < nchunks)
                    process(rb, c + 1);
            }
            if (nchunks == 0) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&acce_bar[acc]));
            }
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1;
            }
            if (++acc == p.n_acc) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    __syncwarp();
    if (threadIdx.x == 0 && *s_abort && p.status)
        atomicOr(p.status, DSA_DEV_TIMEOUT);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1)
        tmem_dealloc(tmem_base, p.n_acc * p.acc_cols);
}

template <int D, int H>
dsa_status launch_fp8_dh(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const dsa_paged_cache* k = a.k;
    const int P = k->page_kv;
    const int G = a.rows_per_unit;
    const int n_cols = ((G * H + 15) / 16) * 16;
    uint32_t acc_cols = 32;
    while (acc_cols < static_cast<uint32_t>(n_cols))
        acc_cols <<= 1;
    const uint32_t q_buf_bytes = ((static_cast<uint32_t>(n_cols) * D + 1023u) / 1024u) * 1024u;

    // tensor maps: K values [num_pages][P][D] bytes, scales [num_pages][P] fp32,
    // q [rows_total*H][D] bytes
    CUtensorMap tm_k, tm_s, tm_q;
    const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : (D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(P),
                                  static_cast<uint64_t>(k->num_pages)};
        const uint64_t strides[2] = {static_cast<uint64_t>(k->val_token_stride),
                                     static_cast<uint64_t>(k->val_page_stride)};
        const uint32_t box[3] = {static_cast<uint32_t>(D), static_cast<uint32_t>(P), 1};
        dsa_status st = encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, k->values, dims, strides, box, sw);
        if (st != DSA_OK)
            return st;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(P), static_cast<uint64_t>(k->num_pages)};
        const uint64_t strides[1] = {static_cast<uint64_t>(k->sc_page_stride)};
        const uint32_t box[2] = {static_cast<uint32_t>(P), 1};
        dsa_status st = encode_tiled(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, k->scales, dims, strides, box,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != DSA_OK)
            return st;
    }
    {
        const uint64_t rows_total = static_cast<uint64_t>(a.batch) * a.next_n * H;
        const uint64_t dims[2] = {static_cast<uint64_t>(D), rows_total};
        const uint64_t strides[1] = {static_cast<uint64_t>(D)};
        const uint32_t box[2] = {static_cast<uint32_t>(D), static_cast<uint32_t>(n_cols)};
        dsa_status st = encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box, sw);
        if (st != DSA_OK)
            return st;
    }

    // as many stages as fit next to the q buffers
    const int budget = std::min(dev.max_smem_optin, 227 * 1024) - 1024;
    // (a multiple of the producer count: each producer owns every kProd-th stage)
    int stages = kMaxStages;
    while (stages > kProd && static_cast<int>(smem_map(D, stages, q_buf_bytes).total) > budget)
        stages -= kProd;
    const SmemMap mp = smem_map(D, stages, q_buf_bytes);
    if (static_cast<int>(mp.total) > budget)
        return DSA_ERR_UNSUPPORTED;
    const int smem_bytes = static_cast<int>(mp.total) + 1024;

    LogitsParams p;
    p.sched = a.sched;
    p.context_lens = a.context_lens;
    p.block_table = k->block_table;
    p.bt_stride = k->bt_row_stride;
    p.max_pages = k->max_pages_per_seq;
    p.num_pages = k->num_pages;
    p.page_kv = P;
    p.next_n = a.next_n;
    p.row_begin = a.row_begin;
    p.row_end = a.row_end;
    p.num_units = a.num_units;
    p.rows_per_unit = G;
    p.weights = a.weights;
    p.logits = a.logits;
    p.logits_stride = a.logits_row_stride;
    p.logits_width = a.logits_width;
    p.status = a.status;
    p.stages = stages;
    p.n_cols = n_cols;
    p.acc_cols = acc_cols;
    p.n_acc = static_cast<int>(std::min<uint32_t>(kMaxAcc, 512u / acc_cols));
    p.q_buf_bytes = q_buf_bytes;

    auto kern = logits_fp8_kernel<D, H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e);
    kern<<<dev.sm_count, kThreads, smem_bytes, stream>>>(tm_k, tm_s, tm_q, p);
    return check_launch();
}

template <int D>
dsa_status launch_fp8_d(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    switch (a.num_heads) {
    case 4: return launch_fp8_dh<D, 4>(a, dev, stream);
    case 8: return launch_fp8_dh<D, 8>(a, dev, stream);
    case 16: return launch_fp8_dh<D, 16>(a, dev, stream);
    case 32: return launch_fp8_dh<D, 32>(a, dev, stream);
    case 64: return launch_fp8_dh<D, 64>(a, dev, stream);
    case 128: return launch_fp8_dh<D, 128>(a, dev, stream);
    default: return DSA_ERR_UNSUPPORTED;
    }
}

}  // namespace

dsa_status launch_logits_fp8(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    switch (a.k->head_dim) {
    case 32: return launch_fp8_d<32>(a, dev, stream);
    case 64: return launch_fp8_d<64>(a, dev, stream);
    case 128: return launch_fp8_d<128>(a, dev, stream);
    default: return DSA_ERR_UNSUPPORTED;
    }
}

}  // namespace dsa
