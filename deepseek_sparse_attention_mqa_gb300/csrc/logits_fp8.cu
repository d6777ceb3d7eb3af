// logits_fp8.cu -- paged lightning-indexer MQA logits over an FP8 (e4m3) K cache.
//
//   logits[r][s] = k_scale[s] * sum_h w[r][h] * relu(q[r][h] . k[s])
//
// Prior art on the pages ("SM120 FP8 paged MQA page 32", vllm-project/DeepGEMM #14,
// Summary and review): one TMA copy per physical page, never a tile that
// straddles two non-contiguous pages (BLOCK_KV = min(PAGE_KV, 64)), several
// TMA warps each owning a KV group, 2-3 stages to fit SM120's 99 KiB.
//
// GB300 design (one persistent CTA per SM, warp-specialised).  The CTA takes an
// equal share of the 128-token tiles and walks it in super-tiles: up to R
// consecutive tiles of one unit (R = 4 at D = 128 and 64 heads, so a stage holds
// up to 64 KB of K and two super-tile accumulators fit in TMEM).  Super-tile j
// (CTA-local ordinal) lives in stage j % stages and accumulator j % n_acc.  Each
// role is split over several warps, because on this part a single thread's chain
// of barrier waits, copy or MMA issues and commits costs more than a tile's HBM
// time:
//   warps 0-3   TMA producers, all on every super-tile: one 3-D box per physical
//               page (lane i of warp w copies page w + 4i) into a 128B/64B/32B-
//               swizzled K-major stage, and the per-token fp32 scales with one
//               16-byte cp.async per lane.
//   warps 4-5   single-thread tcgen05.mma issuers (super-tile j -> warp j % 2),
//               kind::f8f6f4: D[128 tokens x N] += K_tile[128 x D] * Q[N x D]^T,
//               N = rows x heads; each TMEM lane is one token and each column
//               one (row, head).  Warp 4 also owns the TMEM allocation.
//   warp 6      q rows + head weights of each unit (TMA / bulk copies into
//               one of two buffers), running up to one unit ahead.
//   warps 7-14  epilogue, 2 warpgroups, super-tile j -> group j % 2:
//               tcgen05.ld of the thread's own lane, then the relu /
//               head-weighting / k_scale reduction is thread-local (no
//               shuffles, rows of a unit past its last row skipped), and each
//               warp stores 32 consecutive logits per row.  A unit of only 4 or
//               8 columns (4 or 8 heads, one row) has those columns of several
//               blocks loaded before one wait.
//   Up to eight TMEM accumulators let the epilogues of earlier super-tiles
//   overlap the MMAs of later ones; the stage ring keeps K bytes in flight.
//   Without a schedule buffer (at most kInlineUnits units) every CTA first
//   builds the unit records in shared memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "fused_topk.cuh"
#include "host.h"
#include "logits_common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kMaxStages = 16;
constexpr int kProd = 4;                  // TMA producer warps: 0 .. kProd-1
constexpr int kMma = 2;                   // MMA issuer warps: kProd .. kProd+kMma-1
constexpr int kQWarp = kProd + kMma;      // q rows + unit weights loader
constexpr int kEpiWarp0 = kQWarp + 1;     // first epilogue warp
constexpr int kPageCache = 128;           // physical page ids cached by each producer warp
constexpr int kMaxAcc = 8;                // TMEM accumulators in flight
constexpr int kMaxR = 8;                  // 128-token tiles per super-tile
// K bytes per stage.  64 KB (4 tiles at D = 128) beats 32 KB by 8 % on the decode
// workload and 13 % on 64 x 128 heads over longer contexts, though only two such
// stages fit: the per-super-tile handshakes are paid over twice the bytes.
constexpr uint32_t kMaxStageKBytes = 65536;

// Epilogue warpgroups and block size per head count.
template <int H>
struct Fp8Roles {
    static constexpr int kGroups = 2;
    static constexpr int kEpiWarps = 4 * kGroups;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
};

struct LogitsParams {
    const int32_t* sched;       // prebuilt schedule, or null: the CTAs build the units themselves
    int batch;
    int inline_units;           // units built in shared memory (0 with a prebuilt schedule)
    const int32_t* context_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    const uint8_t* scales;      // fp32 per token, page stride sc_page_stride bytes
    int64_t sc_page_stride;
    int max_pages;
    int num_pages;
    int page_kv;
    int next_n;
    int ratio;          // tokens per K-cache entry
    int row_begin;
    int row_end;
    int num_units;
    int rows_per_unit;
    const float* weights;
    float* logits;
    int64_t logits_stride;
    int logits_width;
    int32_t* status;
    int R;              // 128-token tiles per super-tile (1, 2, 4 or 8)
    int stages;         // super-tile stages (multiple of kMma and n_grp)
    int n_cols;         // MMA N (multiple of 16)
    int w_cols;         // n_cols rounded up to the 32-column epilogue chunk
    uint32_t acc_cols;  // TMEM columns per 128-token block (power of two >= 32, >= n_cols)
    int n_acc;          // super-tile accumulators (n_acc * R * acc_cols <= 512)
    int n_grp;          // active epilogue warpgroups (divides n_acc)
    uint32_t q_buf_bytes;
    FusedTopk topk;     // fused top-k outputs (kernels instantiated with kFuse)
};

template <int D>
struct Fp8Tile {
    static constexpr uint32_t kBlockBytes = kTileTokens * D;   // K bytes of one 128-token block
    static constexpr uint32_t kLayout = D == 128 ? kLayoutSw128 : (D == 64 ? kLayoutSw64 : kLayoutSw32);
    static constexpr uint32_t kSbo = 8 * D;                    // 8 rows per swizzle atom
    static constexpr int kKSteps = D / 32;                      // K = 32 bytes per MMA
};

// Shared memory map (offsets from a 1024-aligned base).
struct SmemMap {
    uint32_t k_off, q_off, sc_off, w_off, ks_off, pc_off, bar_off, misc_off, units_off, total;
};

__host__ __device__ __forceinline__ SmemMap smem_map(int D, int R, int stages, uint32_t q_buf_bytes, int w_cols,
                                                     int epi_warps, int inline_units)
{
    SmemMap m;
    m.k_off = 0;
    m.q_off = m.k_off + stages * R * kTileTokens * D;
    m.sc_off = m.q_off + 2 * q_buf_bytes;
    m.w_off = m.sc_off + stages * R * kTileTokens * 4;
    m.ks_off = m.w_off + 2 * w_cols * 4;                     // unit weights, one slot per q buffer
    m.pc_off = m.ks_off + epi_warps * R * 32 * 4;            // token scales per epilogue warp
    m.bar_off = m.pc_off + kProd * kPageCache * 4;
    m.misc_off = m.bar_off + (2 * kMaxStages + 2 * kMaxAcc + 4 + kMma) * 8;
    m.units_off = m.misc_off + 16;               // inline schedule: records, then scan scratch
    m.total = m.units_off + (inline_units > 0 ? inline_units * 32 + kInlineScratchBytes : 0);
    return m;
}

template <int D, int H, bool kFuse>
__global__ void __launch_bounds__(Fp8Roles<H>::kThreads, 1)
logits_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const LogitsParams p)
{
    using T = Fp8Tile<D>;
    constexpr int kEpiWarps = Fp8Roles<H>::kEpiWarps;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemMap mp = smem_map(D, p.R, p.stages, p.q_buf_bytes, p.w_cols, kEpiWarps, p.inline_units);
    const uint32_t stage_bytes = static_cast<uint32_t>(p.R) * T::kBlockBytes;
    const int stage_tokens = p.R * kTileTokens;
    uint8_t* sK = smem + mp.k_off;
    uint8_t* sQ = smem + mp.q_off;
    float* sS = reinterpret_cast<float*>(smem + mp.sc_off);
    float* sW = reinterpret_cast<float*>(smem + mp.w_off);       // [2][w_cols] unit weights
    float* sKs = reinterpret_cast<float*>(smem + mp.ks_off);
    int* s_pages = reinterpret_cast<int*>(smem + mp.pc_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + mp.bar_off);
    uint64_t* full_bar = bars;                       // [stages]
    uint64_t* empty_bar = bars + kMaxStages;         // [stages]
    uint64_t* accf_bar = bars + 2 * kMaxStages;      // [kMaxAcc]
    uint64_t* acce_bar = accf_bar + kMaxAcc;         // [kMaxAcc]
    uint64_t* qf_bar = acce_bar + kMaxAcc;           // [2]
    uint64_t* qe_bar = qf_bar + 2;                   // [2]
    uint64_t* done_bar = qe_bar + 2;                 // [kMma]
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(smem + mp.misc_off);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + mp.misc_off + 4);
    volatile int* s_u0 = reinterpret_cast<volatile int*>(smem + mp.misc_off + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the next kernel (the top-k, launched as a programmatic dependent) may
    // start its prologue on SMs this grid frees; it waits for the logits
    pdl_launch_dependents();

    // ---- the schedule: a prebuilt buffer (its header checked, uniformly over the
    // CTA, before any allocation) or the units built here in shared memory
    const SchedUnit* units;
    int total_tiles;
    if (p.sched) {
        const int32_t* hdr = p.sched;
        units = reinterpret_cast<const SchedUnit*>(p.sched + kSchedHeaderWords);
        if (hdr[0] != kSchedMagic || hdr[1] != p.num_units || hdr[2] != p.rows_per_unit ||
            hdr[3] != p.row_begin || hdr[4] != p.row_end || hdr[5] != p.next_n || hdr[7] != p.ratio) {
            if (threadIdx.x == 0 && p.status)
                atomicOr(p.status, DSA_DEV_SCHEDULE);
            return;
        }
        total_tiles = hdr[6];
    } else {
        SchedUnit* su = reinterpret_cast<SchedUnit*>(smem + mp.units_off);
        int* scratch = reinterpret_cast<int*>(smem + mp.units_off + p.inline_units * 32);
        total_tiles = build_inline_units(su, scratch, p.context_lens, p.batch, p.next_n, p.ratio, p.rows_per_unit,
                                         p.row_begin, p.row_end, p.num_units,
                                         blockIdx.x == 0 ? p.status : nullptr);
        units = su;
    }
    const int t0 = static_cast<int>((static_cast<long long>(blockIdx.x) * total_tiles) / gridDim.x);
    const int t1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * total_tiles) / gridDim.x);
    // the fused top-k phase's view of this launch (its shared memory is the
    // scoring stages', free once the CTA's tiles are done)
    auto phase_args = [&](bool has_tiles, int u0) {
        FusedPhaseArgs fa;
        fa.units = units;
        fa.num_units = p.num_units;
        fa.total_tiles = total_tiles;
        fa.t0 = t0;
        fa.t1 = t1;
        fa.R = p.R;
        fa.u0 = u0;
        fa.has_tiles = has_tiles;
        fa.logits = p.logits;
        fa.logits_stride = p.logits_stride;
        fa.logits_width = p.logits_width;
        fa.next_n = p.next_n;
        fa.ratio = p.ratio;
        fa.row_begin = p.row_begin;
        fa.context_lens = p.context_lens;
        fa.status = p.status;
        fa.smem = smem;
        fa.smem_bytes = mp.bar_off;
        return fa;
    };
    if (t0 >= t1 || p.num_units == 0) {
        if constexpr (kFuse)
            fused_topk_phase(phase_args(false, 0), p.topk);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), kProd);     // one arrive (with its TMA bytes) per producer warp
            mbar_init(smem_u32(&empty_bar[s]), 1 + 4);   // MMA commit + the super-tile's 4 epilogue warps
        }
        for (int a = 0; a < kMaxAcc; ++a) {
            mbar_init(smem_u32(&accf_bar[a]), 1);
            mbar_init(smem_u32(&acce_bar[a]), 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&qf_bar[a]), 1);
            // every MMA warp and every active epilogue warp has finished with the unit
            mbar_init(smem_u32(&qe_bar[a]), kMma + 4 * p.n_grp);
        }
        for (int a = 0; a < kMma; ++a)
            mbar_init(smem_u32(&done_bar[a]), 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_q);
    }
    if (warp == kProd) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), p.n_acc * p.R * p.acc_cols);
        tmem_relinquish();
    }
    if (warp == kProd + 1) {
        const int u0 = find_unit_warp(units, p.num_units, t0);
        if (lane == 0)
            *s_u0 = u0;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const int u0 = *s_u0;                            // the unit of tile t0
    const uint32_t acc_stride = static_cast<uint32_t>(p.R) * p.acc_cols;   // TMEM columns per super-tile
    const WalkParams wp{p.context_lens, p.next_n, p.num_units};
    const int P = p.page_kv;
    const int pages_per_tile = kTileTokens / P;

    if (warp < kProd) {
        // =========================== TMA producers ==========================
        // All kProd producer warps issue every super-tile together: warp pi
        // copies the pages jp with jp % kProd == pi (one lane per page, one TMA
        // box each) and the token scales of the 128-token blocks m with
        // m % kProd == pi, so the serial issue latency of the boxes is split
        // kProd ways.  Each warp arrives once on the stage's full barrier
        // (count kProd) with the bytes of its own boxes.  Physical page ids are
        // fetched by all 32 lanes at once into the warp's own shared-memory
        // cache.
        const int pi = warp;
        int* my_pages = s_pages + pi * kPageCache;
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, p.R, u0);
        long long issued = 0;
        int pc_unit = -1, pc_lp0 = 0, pc_cnt = 0;
        int stage = 0;
        uint32_t phase = 0;
        for (int j = 0; w.valid(); ++j, w.next()) {
            if (__any_sync(0xffffffffu, *s_abort))
                break;
            int ok = 1;
            const UnitInfo& ui = w.w.ui;
            const int lp_first = w.tile_in_unit() * pages_per_tile;
            const int npages = w.nt * pages_per_tile;
            if (w.w.u != pc_unit || lp_first + npages > pc_lp0 + pc_cnt) {
                // refill: this unit's pages from lp_first up to what this CTA will use
                const int tiles_here = min(t1 + p.R - 1, ui.tile_end) - ui.tile_begin;
                const int lp_vis = (ui.vis_max + P - 1) / P;
                const int lp_end = min(tiles_here * pages_per_tile, lp_vis);
                const int cnt = min(kPageCache, max(lp_end - lp_first, npages));
                __syncwarp();
                // every load of the refill in flight before any store: one
                // global-memory latency per refill instead of one per 32 pages
                int pgv[kPageCache / 32];
#pragma unroll
                for (int k = 0; k < kPageCache / 32; ++k) {
                    const int i = lane + 32 * k, lp = lp_first + i;
                    pgv[k] = (i < cnt && lp < lp_vis && lp < p.max_pages)
                                 ? __ldg(p.block_table + static_cast<int64_t>(ui.seq) * p.bt_stride + lp)
                                 : -1;
                }
#pragma unroll
                for (int k = 0; k < kPageCache / 32; ++k)
                    if (lane + 32 * k < cnt)
                        my_pages[lane + 32 * k] = pgv[k];
                __syncwarp();
                pc_unit = w.w.u;
                pc_lp0 = lp_first;
                pc_cnt = cnt;
            }
            if (lane == 0 && ok)
                ok = mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0)
                    *s_abort = 1;
                break;
            }
            // This warp's share: per owned 128-token block m, lane l copies the
            // fp32 scales of tokens [4l, 4l + 4) with one 16-byte cp.async
            // (tracked by the full barrier through cp.async.mbarrier.arrive),
            // and lane i issues the TMA box of page pi + i * kProd.  The
            // cp.async arrivals are registered before the warp's own arrive, and
            // the expected TMA bytes before any box is issued, so the phase
            // cannot complete early.
            const uint32_t fb = smem_u32(&full_bar[stage]);
            auto page_of = [&](int jp) -> int {
                const int lp = lp_first + jp;
                if (lp * P >= ui.vis_max)
                    return -1;                             // past the visible length: not loaded
                const int pg = my_pages[lp - pc_lp0];
                return (pg >= 0 && pg < p.num_pages) ? pg : -2;
            };
            for (int m = pi; m < w.nt; m += kProd) {
                const int tok0 = m * kTileTokens + lane * 4;
                const int pg = page_of(tok0 / P);
                if (pg >= 0)
                    cp_async_16(smem_u32(sS + stage * stage_tokens + tok0),
                                p.scales + static_cast<int64_t>(pg) * p.sc_page_stride + (tok0 % P) * 4);
            }
            cp_async_mbar_arrive(fb);
            const int jp = pi + lane * kProd;
            const int pg_k = jp < npages ? page_of(jp) : -1;
            if (pg_k == -2 && p.status)
                atomicOr(p.status, DSA_DEV_BAD_PAGE);
            const uint32_t kmask = __ballot_sync(0xffffffffu, pg_k >= 0);
            __syncwarp();
            if (lane == 0)
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(__popc(kmask)) * static_cast<uint32_t>(P) * D);
            __syncwarp();
            if (pg_k >= 0)
                tma_load_3d(smem_u32(sK + stage * stage_bytes + jp * P * D), &tm_k, fb, 0, 0, pg_k);
            ++issued;
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        // drain: every copy this warp issued has landed before the CTA exits
        // (a stage is reissued only after its previous contents were consumed,
        // so only the last `stages` super-tiles may still be in flight)
        if (lane == 0) {
            const long long lo = issued > p.stages ? issued - p.stages : 0;
            for (long long jj = lo; jj < issued; ++jj)
                mbar_wait(smem_u32(&full_bar[jj % p.stages]), static_cast<uint32_t>((jj / p.stages) & 1));
        }
    } else if (warp == kQWarp) {
        // ======================= q rows + unit weights ======================
        // Runs ahead of the MMA warps by up to one unit: as soon as a q buffer
        // is released (qe: its unit's MMAs and epilogues are done), the next
        // unit's q rows ([rows x heads, D]) and head weights ([rows x heads]
        // fp32, zero-padded to w_cols) are copied into it.
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, p.R, u0);
        int ucount = 0, unit = -1;
        bool ok = true;
        for (; w.valid(); w.next()) {
            if (w.w.u == unit)
                continue;
            unit = w.w.u;
            const UnitInfo& ui = w.w.ui;
            const int qb = ucount & 1;
            if (lane == 0)
                ok = mbar_wait(smem_u32(&qe_bar[qb]), ((ucount >> 1) & 1) ^ 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || *s_abort)
                break;
            const int nw = ui.nrows * H;
            float* wdst = sW + qb * p.w_cols;
            for (int c = nw + lane; c < p.w_cols; c += 32)
                wdst[c] = 0.f;
            __syncwarp();
            if (lane == 0) {
                const uint32_t qfb = smem_u32(&qf_bar[qb]);
                mbar_arrive_expect_tx(qfb, static_cast<uint32_t>(p.n_cols) * D + static_cast<uint32_t>(nw) * 4u);
                tma_load_2d(smem_u32(sQ + qb * p.q_buf_bytes), &tm_q, qfb, 0, ui.first_row * H);
                bulk_load(smem_u32(wdst), p.weights + static_cast<int64_t>(ui.first_row) * H,
                          static_cast<uint32_t>(nw) * 4u, qfb);
            }
            ++ucount;
        }
        if (lane == 0) {
            if (!ok)
                *s_abort = 1;
            // drain: the last (at most two) copies have landed before the CTA exits
            for (int u = ucount > 2 ? ucount - 2 : 0; u < ucount; ++u)
                mbar_wait(smem_u32(&qf_bar[u & 1]), static_cast<uint32_t>((u >> 1) & 1));
        }
    } else if (warp < kQWarp) {
        // =========================== MMA issuers ============================
        // Warp mi issues the super-tiles with j % kMma == mi: per 128-token
        // block m, D[acc + m * acc_cols] = K_block_m Q^T over D / 32 k-steps.
        // Every MMA warp walks all super-tiles to follow the unit changes: each
        // waits for the unit's q rows and commits the unit's q buffer release
        // (qe counts kMma commits), so the buffer is reloaded only after the
        // MMAs of all of them have read it.  stages and n_acc are multiples of
        // kMma, so a stage or an accumulator is only ever used by one warp.
        const int mi = warp - kProd;
        if (lane == 0) {
            const uint32_t idesc = make_idesc(0, 0, 0, 128, static_cast<uint32_t>(p.n_cols));
            SuperWalk w;
            w.start(wp, units, total_tiles, t0, t1, p.R, u0);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            int ucount = 0, qb = 0, unit = -1;
            bool ok = true;
            for (int j = 0; w.valid() && !*s_abort; ++j) {
                if (w.w.u != unit) {
                    unit = w.w.u;
                    qb = ucount & 1;
                    if (!mbar_wait(smem_u32(&qf_bar[qb]), (ucount >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    ++ucount;
                }
                if (j % kMma == mi) {
                    if (!mbar_wait(smem_u32(&acce_bar[acc]), acc_phase ^ 1) ||
                        !mbar_wait(smem_u32(&full_bar[stage]), phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc) * acc_stride;
                    const uint32_t a0 = smem_u32(sK + stage * stage_bytes);
                    const uint32_t b_base = smem_u32(sQ + qb * p.q_buf_bytes);
                    for (int m = 0; m < w.nt; ++m) {
#pragma unroll
                        for (int k = 0; k < T::kKSteps; ++k) {
                            const uint64_t ad = make_smem_desc(a0 + m * T::kBlockBytes + k * 32, 16, T::kSbo, T::kLayout);
                            const uint64_t bd = make_smem_desc(b_base + k * 32, 16, T::kSbo, T::kLayout);
                            umma_f8f6f4(d0 + m * p.acc_cols, ad, bd, idesc, k > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(smem_u32(&empty_bar[stage]));
                    umma_commit(smem_u32(&accf_bar[acc]));
                }
                const int u_now = w.w.u;
                w.next();
                if (!w.valid() || w.w.u != u_now)
                    umma_commit(smem_u32(&qe_bar[qb]));    // last super-tile of this unit here
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++acc == p.n_acc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok)
                *s_abort = 1;
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(smem_u32(&done_bar[mi]));
            mbar_wait(smem_u32(&done_bar[mi]), 0);
        }
    } else {
        // =========================== epilogue ===============================
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const int group = ew >> 2;                    // takes the super-tiles with j % n_grp == group
        const int tok = quarter * 32 + lane;          // token of this thread within each 128-token block
        float* myks = sKs + ew * p.R * 32;            // this warp's token scales of the current super-tile
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, p.R, u0);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        int nchunks = 0, L = 0, i0 = 0, unit = -1, ucount = 0, qb = 0;
        const float* wS = sW;                         // the current unit's head weights
        for (int j = 0; w.valid() && group < p.n_grp && !__any_sync(0xffffffffu, *s_abort); ++j) {
            const UnitInfo& ui = w.w.ui;
            if (w.w.u != unit) {
                unit = w.w.u;
                qb = ucount & 1;
                // the unit's weights arrive with its q rows
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&qf_bar[qb]), (ucount >> 1) & 1))) {
                    *s_abort = 1;
                    break;
                }
                ++ucount;
                wS = sW + qb * p.w_cols;
                nchunks = (ui.nrows * H + 31) / 32;
                L = ui.ctx_len;
                i0 = ui.first_row - ui.seq * p.next_n;
                if (lane == 0 && ew == 0 && p.status &&
                    visible_entries(L, p.next_n, i0 + ui.nrows - 1, p.ratio) > p.logits_width)
                    atomicOr(p.status, DSA_DEV_WIDTH);
            }
            if (j % p.n_grp == group) {
            // the token scales are read as soon as the stage has landed, and the
            // stage released, before the MMAs are waited for
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[stage]), phase))) {
                *s_abort = 1;
                break;
            }
            // this thread's token scales move to the warp's own scratch before the
            // stage is released
            const int nt = w.nt;
            for (int m = 0; m < nt; ++m)
                myks[m * 32 + lane] = sS[stage * stage_tokens + m * kTileTokens + tok];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&empty_bar[stage]));
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&accf_bar[acc]), acc_phase))) {
                *s_abort = 1;
                break;
            }
            tc_fence_after_sync();

            const int s_base = w.tile_in_unit() * kTileTokens + tok;
            const uint32_t acc_base = tmem_base + static_cast<uint32_t>(acc) * acc_stride +
                                      (static_cast<uint32_t>(quarter * 32) << 16);
            // Few heads: a unit of 4 columns (4 heads, one row) or 8 (8 heads, one
            // row) has the columns of up to 8 or 4 of its 128-token blocks loaded
            // before one wait -- one TMEM round trip per 32 registers instead of one
            // per block.  Wider units take the per-block path below.
            int m_first = 0;
            if constexpr (H <= 8) {
                const int ucols = ui.nrows * H;
                auto batched = [&](auto width_tag, int cbase, bool last_window) {
                    constexpr int W = decltype(width_tag)::value;
                    constexpr int kBlocks = 32 / W;      // blocks per wait (32 registers)
                    constexpr int kRows = W / H;         // unit rows in the W columns
                    const int ib = cbase / H;            // first row of the window
                    // per row: head weights, visible length and output row (kept in
                    // registers for windows of at most two rows, else read per block)
                    constexpr bool kHoist = kRows <= 2;
                    constexpr int kHr = kHoist ? kRows : 1;
                    float wr[kHr][H];
                    int vis[kHr];
                    float* orow[kHr];
                    auto row_vis = [&](int i) -> int {
                        const int row = ib + i;
                        return row < ui.nrows ? min(visible_entries(L, p.next_n, i0 + row, p.ratio), p.logits_width) : 0;
                    };
                    auto row_out = [&](int i) -> float* {
                        return p.logits + static_cast<int64_t>(ui.first_row + ib + i - p.row_begin) * p.logits_stride;
                    };
                    if constexpr (kHoist) {
#pragma unroll
                        for (int i = 0; i < kRows; ++i) {
#pragma unroll
                            for (int hh = 0; hh < H; ++hh)
                                wr[i][hh] = wS[cbase + i * H + hh];
                            vis[i] = row_vis(i);
                            orow[i] = row_out(i);
                        }
                    }
                    for (int m0 = 0; m0 < nt; m0 += kBlocks) {
                        uint32_t r[kBlocks][W];
#pragma unroll
                        for (int mm = 0; mm < kBlocks; ++mm) {
                            if (m0 + mm < nt) {
                                const uint32_t ta = acc_base + (m0 + mm) * p.acc_cols + cbase;
                                if constexpr (W == 4)
                                    tmem_ld_32x32b_x4(ta, r[mm]);
                                else if constexpr (W == 8)
                                    tmem_ld_32x32b_x8(ta, r[mm]);
                                else if constexpr (W == 16)
                                    tmem_ld_32x32b_x16(ta, r[mm]);
                                else
                                    tmem_ld_32x32b_x32(ta, r[mm]);
                            }
                        }
                        tmem_ld_wait();
                        if (last_window && m0 + kBlocks >= nt) {
                            // the last TMEM reads of this accumulator are in registers
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(smem_u32(&acce_bar[acc]));
                        }
#pragma unroll
                        for (int mm = 0; mm < kBlocks; ++mm) {
                            if (m0 + mm >= nt)
                                break;
                            const int s = s_base + (m0 + mm) * kTileTokens;
                            const float ks = myks[(m0 + mm) * 32 + lane];
#pragma unroll
                            for (int i = 0; i < kRows; ++i) {
                                if (!kHoist && ib + i >= ui.nrows)
                                    break;
                                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                                for (int hh = 0; hh < H; hh += 2) {
                                    const float w0 = kHoist ? wr[kHoist ? i : 0][hh] : wS[cbase + i * H + hh];
                                    const float w1 = kHoist ? wr[kHoist ? i : 0][hh + 1] : wS[cbase + i * H + hh + 1];
                                    a0 = fmaf(w0, fmaxf(__uint_as_float(r[mm][i * H + hh]), 0.f), a0);
                                    a1 = fmaf(w1, fmaxf(__uint_as_float(r[mm][i * H + hh + 1]), 0.f), a1);
                                }
                                const int v = kHoist ? vis[kHoist ? i : 0] : row_vis(i);
                                if (s < v)
                                    (kHoist ? orow[kHoist ? i : 0] : row_out(i))[s] = ks * (a0 + a1);
                            }
                        }
                    }
                };
                if constexpr (H <= 4) {
                    if (ucols <= 4) {
                        batched(std::integral_constant<int, 4>{}, 0, true);
                        m_first = nt;                  // every block done
                    }
                }
                if (H == 8 && m_first == 0 && ucols <= 8) {
                    batched(std::integral_constant<int, 8>{}, 0, true);
                    m_first = nt;
                }
            }
#pragma unroll 1
            for (int m = m_first; m < nt; ++m) {
                const int s = s_base + m * kTileTokens;
                const float ks = myks[m * 32 + lane];
                const uint32_t t_acc = acc_base + m * p.acc_cols;
                // store one finished logit of unit row i
                auto emit = [&](int i, float v) {
                    if (i < ui.nrows) {
                        const int vis = min(visible_entries(L, p.next_n, i0 + i, p.ratio), p.logits_width);
                        if (s < vis)
                            p.logits[static_cast<int64_t>(ui.first_row + i - p.row_begin) * p.logits_stride + s] =
                                ks * v;
                    }
                };
                float cur = 0.f;                       // running row sum (H >= 32)
                auto process = [&](const uint32_t (&r)[32], int c) {
                    const float4* w4 = reinterpret_cast<const float4*>(wS + c * 32);
                    if constexpr (H >= 32) {
                        // one row per chunk: 8 independent partial sums in 4 packed
                        // pairs, one packed FMA per two heads (the relu stays two maxes)
                        uint64_t part[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            part[q] = 0ull;
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            const float4 wv = w4[q4];
                            const uint64_t a01 = pack_f32x2(fmaxf(__uint_as_float(r[4 * q4 + 0]), 0.f),
                                                            fmaxf(__uint_as_float(r[4 * q4 + 1]), 0.f));
                            const uint64_t a23 = pack_f32x2(fmaxf(__uint_as_float(r[4 * q4 + 2]), 0.f),
                                                            fmaxf(__uint_as_float(r[4 * q4 + 3]), 0.f));
                            part[(2 * q4) & 3] = fma_f32x2(pack_f32x2(wv.x, wv.y), a01, part[(2 * q4) & 3]);
                            part[(2 * q4 + 1) & 3] = fma_f32x2(pack_f32x2(wv.z, wv.w), a23, part[(2 * q4 + 1) & 3]);
                        }
                        const float2 p0 = unpack_f32x2(part[0]), p1 = unpack_f32x2(part[1]);
                        const float2 p2 = unpack_f32x2(part[2]), p3 = unpack_f32x2(part[3]);
                        cur += ((p0.x + p0.y) + (p1.x + p1.y)) + ((p2.x + p2.y) + (p3.x + p3.y));
                        if (((c + 1) * 32) % H == 0) {
                            emit((c * 32) / H, cur);
                            cur = 0.f;
                        }
                    } else {
                        // 32 / H rows per chunk, each summed over its H columns; rows
                        // past the unit's last row are skipped (warp-uniform)
                        constexpr int kRowsPerChunk = 32 / H;
                        const int nv = ui.nrows - c * kRowsPerChunk;
                        auto one_row = [&](int i) {          // i is a constant after unrolling
                            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                            for (int hh = 0; hh < H; hh += 2) {
                                acc0 = fmaf(wS[c * 32 + i * H + hh], fmaxf(__uint_as_float(r[i * H + hh]), 0.f), acc0);
                                acc1 = fmaf(wS[c * 32 + i * H + hh + 1], fmaxf(__uint_as_float(r[i * H + hh + 1]), 0.f), acc1);
                            }
                            emit(c * kRowsPerChunk + i, acc0 + acc1);
                        };
                        // One valid row (every decode unit at next_n = 1) is the common
                        // case: a straight line.  Written as the guarded loop alone, the
                        // compiler predicates all 32 / H row bodies and runs them for
                        // every block (measured: ~700 cycles per block at 4 heads).
                        if (nv == 1) {
                            one_row(0);
                        } else {
#pragma unroll
                            for (int i = 0; i < kRowsPerChunk; ++i) {
                                if (i >= nv)
                                    break;
                                one_row(i);
                            }
                        }
                    }
                };
                // two 32-column TMEM loads in flight per round, one at H <= 8
                // (units wider than 8 columns; the registers go to the batched
                // path above)
                constexpr int kPerRound = H <= 8 ? 1 : 2;
                for (int c = 0; c < nchunks; c += kPerRound) {
                    uint32_t r[kPerRound][32];
                    tmem_ld_32x32b_x32(t_acc + c * 32, r[0]);
                    if constexpr (kPerRound == 2) {
                        if (c + 1 < nchunks)
                            tmem_ld_32x32b_x32(t_acc + (c + 1) * 32, r[kPerRound - 1]);
                    }
                    tmem_ld_wait();
                    if (m + 1 == nt && c + kPerRound >= nchunks) {
                        // last TMEM reads of this accumulator are in registers: release it early
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(smem_u32(&acce_bar[acc]));
                    }
                    process(r[0], c);
                    if constexpr (kPerRound == 2) {
                        if (c + 1 < nchunks)
                            process(r[kPerRound - 1], c + 1);
                    }
                }
            }
            if (nchunks == 0) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&acce_bar[acc]));
            }
            }
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1;
            }
            if (++acc == p.n_acc) {
                acc = 0;
                acc_phase ^= 1;
            }
            // past the unit's last super-tile here: this warp is done with its
            // q buffer and weights
            const int u_now = w.w.u;
            w.next();
            if (!w.valid() || w.w.u != u_now) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&qe_bar[qb]));
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // every role is done: a wait that gave up anywhere in the CTA is visible now
    if (threadIdx.x == 0 && *s_abort && p.status)
        atomicOr(p.status, DSA_DEV_TIMEOUT);
    if (warp == kProd)
        tmem_dealloc(tmem_base, p.n_acc * p.R * p.acc_cols);
    if constexpr (kFuse) {
        // outputs are invalid after a timeout (DSA_DEV_TIMEOUT is set): no selection
        if (!*s_abort)
            fused_topk_phase(phase_args(true, u0), p.topk);
    }
}

constexpr int lcm2(int a, int b)
{
    int x = a, y = b;
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return a / x * b;
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
    const int w_cols = ((n_cols + 31) / 32) * 32;

    // tensor maps: K values [num_pages][P][D] bytes, q [rows_total*H][D] bytes
    // (the fp32 token scales are copied with cp.async)
    CUtensorMap tm_k, tm_q;
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
        const uint64_t rows_total = static_cast<uint64_t>(a.batch) * a.next_n * H;
        const uint64_t dims[2] = {static_cast<uint64_t>(D), rows_total};
        const uint64_t strides[1] = {static_cast<uint64_t>(D)};
        const uint32_t box[2] = {static_cast<uint32_t>(D), static_cast<uint32_t>(n_cols)};
        dsa_status st = encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box, sw);
        if (st != DSA_OK)
            return st;
    }

    // Super-tile size: as many 128-token tiles as keep a stage within 64 KB of K
    // and two super-tile accumulators within the 512 TMEM columns (at most 8).
    int R = kMaxR;
    while (R > 1 && (static_cast<uint32_t>(R) * kTileTokens * D > kMaxStageKBytes || R * acc_cols > 256u))
        R >>= 1;
    const int n_acc = static_cast<int>(std::min<uint32_t>(kMaxAcc, 512u / (static_cast<uint32_t>(R) * acc_cols)));
    const int n_grp = std::min(Fp8Roles<H>::kGroups, n_acc);
    // As many stages as fit next to the q buffers, a multiple of the MMA-warp
    // and epilogue-group counts (each stage then has one owner of each kind, so
    // no barrier is waited on by a role that lags a full phase behind).
    const int step = lcm2(kMma, n_grp);
    const int budget = std::min(dev.max_smem_optin, 227 * 1024) - 1024;
    constexpr int kEpiWarps = Fp8Roles<H>::kEpiWarps;
    int stages = (kMaxStages / step) * step;
    const int inline_units = a.sched ? 0 : a.num_units;
    while (stages > step &&
           static_cast<int>(smem_map(D, R, stages, q_buf_bytes, w_cols, kEpiWarps, inline_units).total) > budget)
        stages -= step;
    const SmemMap mp = smem_map(D, R, stages, q_buf_bytes, w_cols, kEpiWarps, inline_units);
    if (static_cast<int>(mp.total) > budget || n_acc % lcm2(kMma, n_grp) != 0)
        return DSA_ERR_UNSUPPORTED;
    if (a.topk.k > 0 && mp.bar_off < fused_phase_min_bytes())
        return DSA_ERR_UNSUPPORTED;
    const int smem_bytes = static_cast<int>(mp.total) + 1024;

    LogitsParams p;
    p.sched = a.sched;
    p.batch = a.batch;
    p.inline_units = inline_units;
    p.context_lens = a.context_lens;
    p.block_table = k->block_table;
    p.bt_stride = k->bt_row_stride;
    p.scales = static_cast<const uint8_t*>(k->scales);
    p.sc_page_stride = k->sc_page_stride;
    p.max_pages = k->max_pages_per_seq;
    p.num_pages = k->num_pages;
    p.page_kv = P;
    p.next_n = a.next_n;
    p.ratio = a.ratio;
    p.row_begin = a.row_begin;
    p.row_end = a.row_end;
    p.num_units = a.num_units;
    p.rows_per_unit = G;
    p.weights = a.weights;
    p.logits = a.logits;
    p.logits_stride = a.logits_row_stride;
    p.logits_width = a.logits_width;
    p.status = a.status;
    p.R = R;
    p.stages = stages;
    p.n_cols = n_cols;
    p.w_cols = w_cols;
    p.acc_cols = acc_cols;
    p.n_acc = n_acc;
    p.n_grp = n_grp;
    p.q_buf_bytes = q_buf_bytes;
    p.topk = a.topk;

    auto kern = a.topk.k > 0 ? logits_fp8_kernel<D, H, true> : logits_fp8_kernel<D, H, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e);
    kern<<<dev.sm_count, Fp8Roles<H>::kThreads, smem_bytes, stream>>>(tm_k, tm_q, p);
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
