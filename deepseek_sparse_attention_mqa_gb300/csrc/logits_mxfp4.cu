// logits_mxfp4.cu -- paged lightning-indexer MQA logits over an MXFP4 K cache.
//
//   logits[r][s] = sum_h w[r][h] * relu( sum_d q[r][h][d] * k[s][d] ),
//   q and k elements = e2m1 * 2^(e - 127) with one ue8m0 exponent per 32 elements.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709): the FP4
// (MXFP4) indexer cache, with the FP4 q riding the FP8 q argument and its scales
// passed alongside; there it is a gfx950-only kernel.  "SM120 FP8 paged MQA page
// 32" (vllm-project/DeepGEMM #14): the FP4 sibling derives BLOCK_KV =
// min(PAGE_KV, 64) so a tile never straddles non-contiguous pages.
//
// GB300 design.  Every e2m1 value is exactly an e4m3 value, so the packed cache
// is widened on chip and fed to the same kind::f8f6f4 tensor-core MMA as the FP8
// path; the ue8m0 block scales stay exact powers of two applied in fp32.  The
// CTA walks its tiles in super-tiles of R consecutive 128-token tiles of one
// unit (as the FP8 kernel does), so the per-handshake costs are paid once per
// R tiles:
//   warps 0-1   TMA producers, both on every super-tile: warp w copies the packed
//               values of pages jp = w (mod 2) (one 3-D box per page, one lane
//               each) into a raw stage; warp 1 also copies the super-tile's
//               ue8m0 exponents, 16 bytes per lane with cp.async;
//   warps 2-3   MMA issuers (super-tile j -> warp j % 2): one M=128 MMA per
//               128-token block and 32-element block (K = 32) into its own TMEM
//               accumulator, so block scales are applied per (token, column,
//               block) afterwards;
//   warps 4-5   converters: widen a raw stage (two tokens per thread and block)
//               into swizzled K-major e4m3 tiles with a byte-permute table and
//               decode the token's block exponents to fp32;
//   warp 6      per unit, running up to one unit ahead: widen the q rows and
//               decode the q exponents and head weights into one of two unit
//               buffers (all global loads of a unit issued before any use);
//   warps 7-14  epilogue, 2 warpgroups (super-tile j -> group j % 2):
//               dot = sum_blk 2^(eq+ek-254) * acc_blk, then relu, head weights,
//               store.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "host.h"
#include "fused_topk.cuh"
#include "logits_common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kProd = 2;              // producer warps 0-1
constexpr int kMma = 2;               // MMA warps 2-3
constexpr int kConv0 = kProd + kMma;  // converter warps 4-5
constexpr int kConvWarps = 2;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kQWarp = kConv0 + kConvWarps;  // q rows, q exponents and weights of each unit: warp 6
constexpr int kEpi0 = kQWarp + 1;     // epilogue warps 7-14
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kMaxRaw = 16;           // raw stages (super-tiles)
constexpr int kMaxConv = 8;           // converted stages
constexpr int kMaxAcc = 8;
constexpr int kMaxR = 4;
constexpr int kPageCache = 128;

struct Mx4Params {
    const int32_t* sched;       // prebuilt schedule, or null: the CTAs build the units themselves
    const int32_t* context_lens;
    int batch;
    int inline_units;           // units built in shared memory (0 with a prebuilt schedule)
    const int32_t* block_table;
    int64_t bt_stride;
    int max_pages;
    int num_pages;
    int page_kv;
    int next_n;
    int ratio;                 // tokens per K-cache entry
    int row_begin;
    int row_end;
    int num_units;
    int rows_per_unit;
    const uint8_t* q;          // packed [R*H][D/2]
    const uint8_t* q_scales;   // [R*H][D/32]
    int64_t q_rows;            // R * H
    const uint8_t* k_scales;   // ue8m0 [num_pages][page_kv][D/32], page stride sc_page_stride
    int64_t sc_page_stride;
    const float* weights;
    float* logits;
    int64_t logits_stride;
    int logits_width;
    int32_t* status;
    int R;                     // 128-token tiles per super-tile
    int raw_stages;
    int conv_stages;           // multiple of n_mma and n_grp
    int n_cols;
    int w_cols;                // n_cols rounded up to 32
    uint32_t acc_cols;         // TMEM columns of one (block, 32-element block) accumulator
    int n_acc;                 // super-tile accumulators
    int n_mma;                 // active MMA warps (divides n_acc)
    int n_grp;                 // active epilogue groups (divides n_acc)
    uint32_t q_buf_bytes;
    FusedTopk topk;            // fused top-k outputs (kernels instantiated with kFuse)
};

template <int D>
struct Mx4Layout {
    static constexpr int kNB = D / 32;                         // blocks (scales) per row
    static constexpr uint32_t kRawK = kTileTokens * D / 2;     // packed bytes per 128 tokens
    static constexpr uint32_t kConvK = kTileTokens * D;        // e4m3 bytes per 128 tokens
    static constexpr uint32_t kLayout = D == 128 ? kLayoutSw128 : kLayoutSw64;
    static constexpr uint32_t kSbo = 8 * D;
};

struct Mx4Smem {
    uint32_t raw_k, raw_sc, conv_k, conv_sc, q, w, sq, ks, qraw, wraw, pc, bar, misc, units, total;
};

template <int D>
__host__ __device__ __forceinline__ Mx4Smem mx4_smem(int R, int raw_stages, int conv_stages, uint32_t q_buf_bytes,
                                                     int w_cols, int inline_units)
{
    using Lt = Mx4Layout<D>;
    Mx4Smem m;
    m.conv_k = 0;                                                   // 1024-aligned tiles first
    m.q = m.conv_k + conv_stages * R * Lt::kConvK;
    m.raw_k = m.q + 2 * q_buf_bytes;
    m.raw_sc = m.raw_k + raw_stages * R * Lt::kRawK;
    m.conv_sc = m.raw_sc + ((raw_stages * R * kTileTokens * Lt::kNB + 15) & ~15);
    m.w = m.conv_sc + conv_stages * R * kTileTokens * Lt::kNB * 4;
    m.sq = m.w + 2 * w_cols * 4;                                    // unit weights, one slot per q buffer
    m.ks = m.sq + 2 * Lt::kNB * w_cols * 4;                         // unit q exponents (fp32), per slot
    m.qraw = m.ks + kEpiWarps * R * Lt::kNB * 32 * 4;               // token exponents per epilogue warp
    m.wraw = m.qraw + 2 * ((w_cols * (D / 2) + 15) & ~15);          // packed q rows of the next units
    m.pc = m.wraw + 2 * w_cols * 4;                                 // fp32 weights of the next units
    m.bar = m.pc + kProd * kPageCache * 4;
    m.misc = m.bar + (2 * kMaxRaw + 2 * kMaxConv + 2 * kMaxAcc + 4 + kMma + 2) * 8;
    m.units = m.misc + 16;                                          // inline schedule: records, scan scratch
    m.total = m.units + (inline_units > 0 ? inline_units * 32 + kInlineScratchBytes : 0);
    return m;
}

// ue8m0 exponent -> fp32 2^(e-127) (e = 0: 2^-127, e = 255: NaN).
__device__ __forceinline__ float ue8m0_to_float(uint32_t e)
{
    return __uint_as_float(e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : (e << 23)));
}

// Eight packed e2m1 values (element j in nibble j) -> eight e4m3 bytes (element
// j in byte j).  Every e2m1 value is an e4m3 value: |x| codes 0..7 map to
// 0x00 0x30 0x38 0x3C 0x40 0x44 0x48 0x4C and the sign moves to bit 7.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8_tab(uint32_t w, uint32_t lo_tab, uint32_t hi_tab)
{
    const uint32_t lo16 = w & 0xFFFFu, hi16 = w >> 16;
    const uint32_t m0 = __byte_perm(lo_tab, hi_tab, lo16 & 0x7777u);
    const uint32_t s0 = __byte_perm(0u, 0x80808080u, (lo16 & 0x8888u) >> 1);
    const uint32_t m1 = __byte_perm(lo_tab, hi_tab, hi16 & 0x7777u);
    const uint32_t s1 = __byte_perm(0u, 0x80808080u, (hi16 & 0x8888u) >> 1);
    return make_uint2(m0 | s0, m1 | s1);
}

__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8(uint32_t w)
{
    return e2m1x8_to_e4m3x8_tab(w, 0x3C383000u, 0x4C484440u);
}

// The byte-permute tables for e2m1 magnitudes (0, 0.5, 1, 1.5, 2, 3, 4, 6) times
// 2^-s, 0 <= s <= 8: every such value is exactly an e4m3 value (normal down to
// 2^-6, then a multiple of 2^-9), codes of magnitudes 0-3 in lo, 4-7 in hi.
__device__ __forceinline__ void e2m1_shifted_tables(int s, uint32_t& lo, uint32_t& hi)
{
    const int kE[8] = {0, -1, 0, 0, 1, 1, 2, 2};      // exponent of each magnitude
    const int kM[8] = {0, 0, 0, 4, 0, 4, 0, 4};       // its 3-bit e4m3 mantissa
    uint32_t t[2] = {0u, 0u};
#pragma unroll
    for (int m = 1; m < 8; ++m) {
        const int e = kE[m] - s;
        const uint32_t code = e >= -6 ? static_cast<uint32_t>(((e + 7) << 3) | kM[m])
                                      : static_cast<uint32_t>((8 + kM[m]) >> (-6 - e));
        t[m >> 2] |= code << (8 * (m & 3));
    }
    lo = t[0];
    hi = t[1];
}

// Widen one packed row (D/2 bytes at src, 16-byte aligned) into row `row` of a
// swizzled K-major e4m3 tile.
// The same with each 32-element block's values times 2^-shift[block] (tables from
// e2m1_shifted_tables).
template <int D>
__device__ __forceinline__ void widen_row_tab(const uint8_t* src, uint8_t* tile, int row,
                                              const uint32_t (&tab)[D / 32][2])
{
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {                 // chunk c lies in block c / 2
        const uint2 pk = *reinterpret_cast<const uint2*>(src + 8 * c);
        const uint2 a = e2m1x8_to_e4m3x8_tab(pk.x, tab[c >> 1][0], tab[c >> 1][1]);
        const uint2 b = e2m1x8_to_e4m3x8_tab(pk.y, tab[c >> 1][0], tab[c >> 1][1]);
        *reinterpret_cast<uint4*>(tile + swizzled_offset(row, c, D)) = make_uint4(a.x, a.y, b.x, b.y);
    }
}

template <int D>
__device__ __forceinline__ void widen_row(const uint8_t* src, uint8_t* tile, int row)
{
    uint4 pk[D / 32];                                  // 16-byte loads: half the shared-memory wavefronts
#pragma unroll
    for (int c = 0; c < D / 32; ++c)                   // two 16-element chunks = 16 packed bytes
        pk[c] = *reinterpret_cast<const uint4*>(src + 16 * c);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        const uint2 a = e2m1x8_to_e4m3x8(pk[c].x);
        const uint2 b = e2m1x8_to_e4m3x8(pk[c].y);
        const uint2 a2 = e2m1x8_to_e4m3x8(pk[c].z);
        const uint2 b2 = e2m1x8_to_e4m3x8(pk[c].w);
        *reinterpret_cast<uint4*>(tile + swizzled_offset(row, 2 * c, D)) = make_uint4(a.x, a.y, b.x, b.y);
        *reinterpret_cast<uint4*>(tile + swizzled_offset(row, 2 * c + 1, D)) = make_uint4(a2.x, a2.y, b2.x, b2.y);
    }
}

template <int D, int H, bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
logits_mxfp4_kernel(const __grid_constant__ CUtensorMap tm_k, const Mx4Params p)
{
    using Lt = Mx4Layout<D>;
    constexpr int NB = Lt::kNB;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Mx4Smem mp = mx4_smem<D>(p.R, p.raw_stages, p.conv_stages, p.q_buf_bytes, p.w_cols, p.inline_units);
    const int R = p.R;
    const int st_tokens = R * kTileTokens;
    uint8_t* sRawK = smem + mp.raw_k;
    uint8_t* sRawS = smem + mp.raw_sc;
    uint8_t* sConvK = smem + mp.conv_k;
    float* sConvS = reinterpret_cast<float*>(smem + mp.conv_sc);
    uint8_t* sQ = smem + mp.q;
    float* sW = reinterpret_cast<float*>(smem + mp.w);        // [2][w_cols]
    float* sSq = reinterpret_cast<float*>(smem + mp.sq);      // [2][NB][w_cols]
    float* sKs = reinterpret_cast<float*>(smem + mp.ks);      // [epi warp][R][NB][32]
    int* s_pages = reinterpret_cast<int*>(smem + mp.pc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + mp.bar);
    uint64_t* rawf = bars;
    uint64_t* rawe = rawf + kMaxRaw;
    uint64_t* convf = rawe + kMaxRaw;
    uint64_t* conve = convf + kMaxConv;
    uint64_t* accf = conve + kMaxConv;
    uint64_t* acce = accf + kMaxAcc;
    uint64_t* qf = acce + kMaxAcc;
    uint64_t* qe = qf + 2;
    uint64_t* done_bar = qe + 2;                         // [kMma]
    uint64_t* qraw_bar = done_bar + kMma;                // [2] staged q rows + weights landed
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(smem + mp.misc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + mp.misc + 4);
    volatile int* s_u0 = reinterpret_cast<volatile int*>(smem + mp.misc + 8);
    volatile uint8_t* s_fold = smem + mp.misc + 12;  // [2] per q buffer: its unit's q exponents are folded

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the next kernel (the top-k, launched as a programmatic dependent) may
    // start its prologue on SMs this grid frees; it waits for the logits
    pdl_launch_dependents();
    // the schedule: a prebuilt buffer (header checked uniformly over the CTA) or
    // the units built here in shared memory
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
        SchedUnit* su = reinterpret_cast<SchedUnit*>(smem + mp.units);
        int* scratch = reinterpret_cast<int*>(smem + mp.units + p.inline_units * 32);
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
        fa.smem_bytes = mp.bar;
        return fa;
    };
    if (t0 >= t1 || p.num_units == 0) {
        if constexpr (kFuse)
            fused_topk_phase(phase_args(false, 0), p.topk);
        return;
    }

    const uint32_t acc_stride = static_cast<uint32_t>(R * NB) * p.acc_cols;   // TMEM columns per super-tile
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.raw_stages; ++s) {
            mbar_init(smem_u32(&rawf[s]), kProd);          // one arrive (with its TMA bytes) per producer warp
            mbar_init(smem_u32(&rawe[s]), kConvWarps);
        }
        for (int s = 0; s < p.conv_stages; ++s) {
            mbar_init(smem_u32(&convf[s]), kConvWarps);
            mbar_init(smem_u32(&conve[s]), 1 + 4);         // MMA commit + the super-tile's epilogue warps
        }
        for (int a = 0; a < kMaxAcc; ++a) {
            mbar_init(smem_u32(&accf[a]), 1);
            mbar_init(smem_u32(&acce[a]), 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&qf[a]), 1);                // the q warp
            mbar_init(smem_u32(&qe[a]), p.n_mma + 4 * p.n_grp);
        }
        for (int a = 0; a < kMma; ++a)
            mbar_init(smem_u32(&done_bar[a]), 1);
        for (int a = 0; a < 2; ++a)
            mbar_init(smem_u32(&qraw_bar[a]), 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_map(&tm_k);
    }
    if (warp == kProd) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), p.n_acc * acc_stride);
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
    const int u0 = *s_u0;
    const WalkParams wp{nullptr, p.next_n, p.num_units};
    const int P = p.page_kv;
    const int ppt = kTileTokens / P;

    if (warp < kProd) {
        // =========================== TMA producers ==========================
        const int pi = warp;
        int* my_pages = s_pages + pi * kPageCache;
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, R, u0);
        long long issued = 0;
        int pc_unit = -1, pc_lp0 = 0, pc_cnt = 0;
        int stage = 0;
        uint32_t phase = 0;
        for (; w.valid(); w.next()) {
            if (__any_sync(0xffffffffu, *s_abort))
                break;
            const UnitInfo& ui = w.w.ui;
            const int lp_first = w.tile_in_unit() * ppt;
            const int npages = w.nt * ppt;
            if (w.w.u != pc_unit || lp_first + npages > pc_lp0 + pc_cnt) {
                const int tiles_here = min(t1 + R - 1, ui.tile_end) - ui.tile_begin;
                const int lp_vis = (ui.vis_max + P - 1) / P;
                const int lp_end = min(tiles_here * ppt, lp_vis);
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
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(smem_u32(&rawe[stage]), phase ^ 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0)
                    *s_abort = 1;
                break;
            }
            auto page_of = [&](int jp) -> int {
                const int lp = lp_first + jp;
                if (lp * P >= ui.vis_max)
                    return -1;                             // past the visible length: not loaded
                const int pg = my_pages[lp - pc_lp0];
                return (pg >= 0 && pg < p.num_pages) ? pg : -2;
            };
            // This warp's share: lane i issues the packed-value box of page
            // pi + 4i; warp 0's lanes also copy the super-tile's exponents (16 bytes
            // each, cp.async tracked by the same full barrier).  The cp.async
            // arrivals are registered before the warp's own arrive and the
            // expected TMA bytes before any box is issued.
            const uint32_t fb = smem_u32(&rawf[stage]);
            if (pi == kProd - 1) {
                const int segs = st_tokens * NB / 16;      // 16-byte exponent segments of a full super-tile
                for (int sg = lane; sg < segs; sg += 32) {
                    const int tok0 = sg * 16 / NB;         // first token of the segment
                    if (tok0 < w.nt * kTileTokens) {
                        const int pg = page_of(tok0 / P);
                        if (pg >= 0)
                            cp_async_16(smem_u32(sRawS + stage * st_tokens * NB + sg * 16),
                                        p.k_scales + static_cast<int64_t>(pg) * p.sc_page_stride + (tok0 % P) * NB);
                    }
                }
                cp_async_mbar_arrive(fb);
            }
            const int jp = pi + lane * kProd;
            const int pg_k = jp < npages ? page_of(jp) : -1;
            if (pg_k == -2 && p.status)
                atomicOr(p.status, DSA_DEV_BAD_PAGE);
            const uint32_t kmask = __ballot_sync(0xffffffffu, pg_k >= 0);
            __syncwarp();
            if (lane == 0)
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(__popc(kmask)) * static_cast<uint32_t>(P) * (D / 2));
            __syncwarp();
            if (pg_k >= 0)
                tma_load_3d(smem_u32(sRawK + stage * R * Lt::kRawK + jp * P * (D / 2)), &tm_k, fb, 0, 0, pg_k);
            ++issued;
            if (++stage == p.raw_stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        // drain: only the last raw_stages super-tiles may still be in flight
        if (lane == 0) {
            const long long lo = issued > p.raw_stages ? issued - p.raw_stages : 0;
            for (long long jj = lo; jj < issued; ++jj)
                mbar_wait(smem_u32(&rawf[jj % p.raw_stages]), static_cast<uint32_t>((jj / p.raw_stages) & 1));
        }
    } else if (warp >= kConv0 && warp < kQWarp) {
        // =========================== converters =============================
        const int ct = threadIdx.x - kConv0 * 32;      // 0..63: tokens ct, ct + 64 of each 128-token block
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, R, u0);
        int rs = 0, cs = 0;
        uint32_t rph = 0, cph = 0;
        for (; w.valid() && !__any_sync(0xffffffffu, *s_abort); w.next()) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&rawf[rs]), rph) &&
                                             mbar_wait(smem_u32(&conve[cs]), cph ^ 1))) {
                *s_abort = 1;
                break;
            }
            for (int m2 = 0; m2 < 2 * w.nt; ++m2) {
                const int m = m2 >> 1, row = (m2 & 1) * kConvThreads + ct;   // row of the 128-token block
                const int t = m * kTileTokens + row;       // token of the super-tile
                widen_row<D>(sRawK + rs * R * Lt::kRawK + t * (D / 2), sConvK + (cs * R + m) * Lt::kConvK, row);
                const uint8_t* sc = sRawS + rs * st_tokens * NB + t * NB;
#pragma unroll
                for (int bk = 0; bk < NB; ++bk)
                    sConvS[(cs * st_tokens + t) * NB + bk] = ue8m0_to_float(sc[bk]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&rawe[rs]));
                mbar_arrive(smem_u32(&convf[cs]));
            }
            if (++rs == p.raw_stages) {
                rs = 0;
                rph ^= 1;
            }
            if (++cs == p.conv_stages) {
                cs = 0;
                cph ^= 1;
            }
        }
    } else if (warp == kQWarp) {
        // ============= q rows, q exponents, head weights of each unit ========
        // The packed q rows and fp32 weights of the next unit are bulk-copied
        // into a staging buffer while this unit's are widened, so a unit change
        // costs one local widening pass, not a chain of global loads.
        uint8_t* sQraw = smem + mp.qraw;
        float* sWraw = reinterpret_cast<float*>(smem + mp.wraw);
        const uint32_t qraw_bytes = (static_cast<uint32_t>(p.w_cols) * (D / 2) + 15u) & ~15u;
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, R, u0);
        // the sequence of this CTA's units (the walk skips super-tiles of the same unit)
        auto stage_unit = [&](const UnitInfo& ui, int slot) {
            const int64_t r0 = static_cast<int64_t>(ui.first_row) * H;
            const uint32_t nvalid = static_cast<uint32_t>(ui.nrows * H);
            const uint32_t bar = smem_u32(&qraw_bar[slot]);
            mbar_arrive_expect_tx(bar, nvalid * (D / 2) + nvalid * 4u);
            bulk_load(smem_u32(sQraw + slot * qraw_bytes), p.q + r0 * (D / 2), nvalid * (D / 2), bar);
            bulk_load(smem_u32(sWraw + slot * p.w_cols), p.weights + r0, nvalid * 4u, bar);
        };
        int ucount = 0, unit = -1;
        bool ok = true;
        SuperWalk ahead = w;                     // walks to the next unit to stage
        if (lane == 0 && w.valid())
            stage_unit(w.w.ui, 0);
        int ahead_unit = w.valid() ? w.w.u : -1;
        for (; w.valid() && ok && !__any_sync(0xffffffffu, *s_abort); w.next()) {
            if (w.w.u == unit)
                continue;
            unit = w.w.u;
            const UnitInfo ui = w.w.ui;
            const int qb = ucount & 1;
            // stage the following unit (its slot was consumed two units ago, by this warp)
            while (ahead.valid() && ahead.w.u == ahead_unit)
                ahead.next();
            if (ahead.valid()) {
                ahead_unit = ahead.w.u;
                if (lane == 0)
                    stage_unit(ahead.w.ui, (ucount + 1) & 1);
            }
            const int64_t r0 = static_cast<int64_t>(ui.first_row) * H;
            const int nvalid = ui.nrows * H;
            // q exponents (ue8m0 codes) straight from global memory (tiny), issued
            // before the waits; column c = lane + 32 k
            uint32_t qc[8][NB];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = lane + 32 * k;
#pragma unroll
                for (int bk = 0; bk < NB; ++bk)
                    qc[k][bk] = (c < p.w_cols && c < nvalid) ? static_cast<uint32_t>(p.q_scales[(r0 + c) * NB + bk])
                                                             : 127u;
            }
            // Folding: each column's blocks are widened times 2^(e_blk - e_max) and
            // its weight times 2^(e_max - 127), so the epilogue drops the per-column
            // scale.  Powers of two scale every product and sum exactly, so the logits
            // are bit-identical, provided nothing leaves the normal range: the unit
            // folds when every code is in [1, 254], a column's codes differ by at most 8
            // (e4m3 holds e2m1 x 2^-8 exactly) and its largest is within 100 of 127.
            uint32_t qmax[8];
            bool fold_ok = true;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t mx = qc[k][0], mn = qc[k][0];
#pragma unroll
                for (int bk = 1; bk < NB; ++bk) {
                    mx = max(mx, qc[k][bk]);
                    mn = min(mn, qc[k][bk]);
                }
                qmax[k] = mx;
                fold_ok = fold_ok && mn >= 1u && mx <= 227u && mx >= 27u && mx - mn <= 8u;
            }
            const bool fold = __all_sync(0xffffffffu, fold_ok);
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&qraw_bar[qb]), (ucount >> 1) & 1) &&
                                             mbar_wait(smem_u32(&qe[qb]), ((ucount >> 1) & 1) ^ 1))) {
                ok = false;
                break;
            }
            uint8_t* qt = sQ + qb * p.q_buf_bytes;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = lane + 32 * k;
                if (rr >= p.n_cols)
                    break;
                if (rr < nvalid) {
                    if (fold) {
                        uint32_t tab[NB][2];
#pragma unroll
                        for (int bk = 0; bk < NB; ++bk)
                            e2m1_shifted_tables(static_cast<int>(qmax[k] - qc[k][bk]), tab[bk][0], tab[bk][1]);
                        widen_row_tab<D>(sQraw + qb * qraw_bytes + rr * (D / 2), qt, rr, tab);
                    } else {
                        widen_row<D>(sQraw + qb * qraw_bytes + rr * (D / 2), qt, rr);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        *reinterpret_cast<uint4*>(qt + swizzled_offset(rr, c, D)) = make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = lane + 32 * k;
                if (c < p.w_cols) {
                    const float wv = c < nvalid ? sWraw[qb * p.w_cols + c] : 0.f;
                    sW[qb * p.w_cols + c] = fold ? wv * ue8m0_to_float(qmax[k]) : wv;
#pragma unroll
                    for (int bk = 0; bk < NB; ++bk)
                        sSq[(qb * NB + bk) * p.w_cols + c] = c < nvalid ? ue8m0_to_float(qc[k][bk]) : 0.f;
                }
            }
            if (lane == 0)
                s_fold[qb] = fold ? 1 : 0;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&qf[qb]));
            ++ucount;
        }
        if (!ok && lane == 0)
            *s_abort = 1;
        // drain: a staged copy that was never consumed has landed before the CTA exits
        if (lane == 0 && ahead_unit != unit && ahead_unit >= 0)
            mbar_wait(smem_u32(&qraw_bar[ucount & 1]), (ucount >> 1) & 1);
    } else if (warp < kConv0) {
        // =========================== MMA issuers ============================
        const int mi = warp - kProd;
        if (lane == 0 && mi < p.n_mma) {
            const uint32_t idesc = make_idesc(0, 0, 0, 128, static_cast<uint32_t>(p.n_cols));
            SuperWalk w;
            w.start(wp, units, total_tiles, t0, t1, R, u0);
            int cs = 0, acc = 0, ucount = 0, qb = 0, unit = -1;
            uint32_t cph = 0, aph = 0;
            bool ok = true;
            for (int j = 0; w.valid() && !*s_abort; ++j) {
                if (w.w.u != unit) {
                    unit = w.w.u;
                    qb = ucount & 1;
                    if (!mbar_wait(smem_u32(&qf[qb]), (ucount >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    ++ucount;
                }
                if (j % p.n_mma == mi) {
                    if (!mbar_wait(smem_u32(&acce[acc]), aph ^ 1) || !mbar_wait(smem_u32(&convf[cs]), cph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t b_base = smem_u32(sQ + qb * p.q_buf_bytes);
                    for (int m = 0; m < w.nt; ++m) {
                        const uint32_t a_base = smem_u32(sConvK + (cs * R + m) * Lt::kConvK);
#pragma unroll
                        for (int bk = 0; bk < NB; ++bk) {
                            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_stride +
                                                    static_cast<uint32_t>(m * NB + bk) * p.acc_cols;
                            const uint64_t ad = make_smem_desc(a_base + bk * 32, 16, Lt::kSbo, Lt::kLayout);
                            const uint64_t bd = make_smem_desc(b_base + bk * 32, 16, Lt::kSbo, Lt::kLayout);
                            umma_f8f6f4(d_tmem, ad, bd, idesc, 0u);
                        }
                    }
                    umma_commit(smem_u32(&conve[cs]));
                    umma_commit(smem_u32(&accf[acc]));
                }
                const int u_now = w.w.u;
                w.next();
                if (!w.valid() || w.w.u != u_now)
                    umma_commit(smem_u32(&qe[qb]));        // past the unit's last super-tile here
                if (++cs == p.conv_stages) {
                    cs = 0;
                    cph ^= 1;
                }
                if (++acc == p.n_acc) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            if (!ok)
                *s_abort = 1;
            umma_commit(smem_u32(&done_bar[mi]));
            mbar_wait(smem_u32(&done_bar[mi]), 0);
        }
    } else {
        // =========================== epilogue ===============================
        const int e = warp - kEpi0;                    // 0..7
        const int quarter = warp & 3;                  // TMEM lanes this warp may access
        const int group = e >> 2;                      // takes the super-tiles with j % n_grp == group
        const int tok = quarter * 32 + lane;
        float* myks = sKs + e * R * NB * 32;           // this warp's token exponents of the super-tile
        SuperWalk w;
        w.start(wp, units, total_tiles, t0, t1, R, u0);
        int cs = 0, acc = 0, ucount = 0, qb = 0, unit = -1;
        uint32_t cph = 0, aph = 0;
        int L = 0, i0 = 0;
        const float* wS = sW;
        const float* sqS = sSq;
        bool folded = false;                           // the unit's q exponents are in its q and weights
        for (int j = 0; w.valid() && group < p.n_grp && !__any_sync(0xffffffffu, *s_abort); ++j) {
            const UnitInfo& ui = w.w.ui;
            if (w.w.u != unit) {
                unit = w.w.u;
                qb = ucount & 1;
                // the unit's weights and q exponents arrive with its q rows
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&qf[qb]), (ucount >> 1) & 1))) {
                    *s_abort = 1;
                    break;
                }
                ++ucount;
                wS = sW + qb * p.w_cols;
                sqS = sSq + qb * NB * p.w_cols;
                folded = s_fold[qb] != 0;
                L = ui.ctx_len;
                i0 = ui.first_row - ui.seq * p.next_n;
                if (e == 0 && lane == 0 && p.status &&
                    visible_entries(L, p.next_n, i0 + ui.nrows - 1, p.ratio) > p.logits_width)
                    atomicOr(p.status, DSA_DEV_WIDTH);
            }
            if (j % p.n_grp == group) {
                // token exponents move to this warp's scratch before the stage is released
                const int nt = w.nt;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&convf[cs]), cph))) {
                    *s_abort = 1;
                    break;
                }
                for (int m = 0; m < nt; ++m)
#pragma unroll
                    for (int bk = 0; bk < NB; ++bk)
                        myks[(m * NB + bk) * 32 + lane] = sConvS[(cs * st_tokens + m * kTileTokens + tok) * NB + bk];
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&conve[cs]));
                // warp-uniform outcome: the TMEM loads below are warp-collective
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&accf[acc]), aph))) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t t_acc0 = tmem_base + static_cast<uint32_t>(acc) * acc_stride +
                                        (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
                for (int m = 0; m < nt; ++m) {
                    const int s = (w.tile_in_unit() + m) * kTileTokens + tok;
                    float sk[NB];
#pragma unroll
                    for (int bk = 0; bk < NB; ++bk)
                        sk[bk] = myks[(m * NB + bk) * 32 + lane];
                    for (int i = 0; i < ui.nrows; ++i) {
                        float rowsum = 0.f;
                        const int c_lo = i * H, c_hi = (i + 1) * H;
                        // 16-column chunks aligned within the accumulator slice (a row of
                        // H < 16 heads lies inside one chunk)
                        for (int cb = c_lo & ~15; cb < c_hi; cb += 16) {
                            float dot[16];
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                dot[q] = 0.f;
                            // two scale blocks' TMEM loads in flight per wait
#pragma unroll
                            for (int b0 = 0; b0 < NB; b0 += 2) {
                                uint32_t r[2][16];
                                tmem_ld_32x32b_x16(t_acc0 + static_cast<uint32_t>(m * NB + b0) * p.acc_cols + cb, r[0]);
                                if (b0 + 1 < NB)
                                    tmem_ld_32x32b_x16(t_acc0 + static_cast<uint32_t>(m * NB + b0 + 1) * p.acc_cols + cb,
                                                       r[1]);
                                tmem_ld_wait();
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    if (b0 + u < NB) {
                                        if (folded) {
#pragma unroll
                                            for (int q = 0; q < 16; ++q)
                                                dot[q] = fmaf(sk[b0 + u], __uint_as_float(r[u][q]), dot[q]);
                                        } else {
                                            const float* sq = sqS + (b0 + u) * p.w_cols + cb;
#pragma unroll
                                            for (int q = 0; q < 16; ++q)
                                                dot[q] = fmaf(sq[q] * sk[b0 + u], __uint_as_float(r[u][q]), dot[q]);
                                        }
                                    }
                                }
                            }
                            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                if (cb + q >= c_lo && cb + q < c_hi)
                                    part[q & 3] = fmaf(wS[cb + q], fmaxf(dot[q], 0.f), part[q & 3]);
                            rowsum += (part[0] + part[1]) + (part[2] + part[3]);
                        }
                        const int vis = min(visible_entries(L, p.next_n, i0 + i, p.ratio), p.logits_width);
                        if (s < vis)
                            p.logits[static_cast<int64_t>(ui.first_row + i - p.row_begin) * p.logits_stride + s] = rowsum;
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&acce[acc]));
            }
            if (++cs == p.conv_stages) {
                cs = 0;
                cph ^= 1;
            }
            if (++acc == p.n_acc) {
                acc = 0;
                aph ^= 1;
            }
            // past the unit's last super-tile here: this warp is done with its buffer
            const int u_now = w.w.u;
            w.next();
            if (!w.valid() || w.w.u != u_now) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&qe[qb]));
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
        tmem_dealloc(tmem_base, p.n_acc * acc_stride);
    if constexpr (kFuse) {
        // outputs are invalid after a timeout (DSA_DEV_TIMEOUT is set): no selection
        if (!*s_abort)
            fused_topk_phase(phase_args(true, u0), p.topk);
    }
}

template <int D, int H>
dsa_status launch_mx4_dh(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    using Lt = Mx4Layout<D>;
    const dsa_paged_cache* k = a.k;
    const int P = k->page_kv;
    const int G = a.rows_per_unit;
    const int n_cols = ((G * H + 15) / 16) * 16;
    const int w_cols = ((n_cols + 31) / 32) * 32;
    uint32_t acc_cols = 32;
    while (acc_cols < static_cast<uint32_t>(n_cols))
        acc_cols <<= 1;
    const uint32_t blk_cols = Lt::kNB * acc_cols;          // TMEM columns of one 128-token block
    if (blk_cols > 512u)
        return DSA_ERR_UNSUPPORTED;
    // super-tile: up to kMaxR tiles while two super-tile accumulators fit in TMEM
    int R = kMaxR;
    while (R > 1 && static_cast<uint32_t>(R) * blk_cols > 256u)
        R >>= 1;
    const int n_acc = static_cast<int>(std::min<uint32_t>(kMaxAcc, 512u / (static_cast<uint32_t>(R) * blk_cols)));
    const int n_mma = std::min(kMma, n_acc);
    const int n_grp = std::min(2, n_acc);
    const uint32_t q_buf_bytes = ((static_cast<uint32_t>(n_cols) * D + 1023u) / 1024u) * 1024u;
    // stage counts: as many as fit, converted stages a multiple of the MMA-warp
    // and epilogue-group counts (each stage then has one owner of each kind)
    const int budget = std::min(dev.max_smem_optin, 227 * 1024) - 1024;
    const int cstep = std::max(n_mma, n_grp);
    int raw_stages = 8, conv_stages = 4;
    const int inline_units = a.sched ? 0 : a.num_units;
    auto fits = [&](int rs, int cs) {
        return static_cast<int>(mx4_smem<D>(R, rs, cs, q_buf_bytes, w_cols, inline_units).total) <= budget;
    };
    while (!fits(raw_stages, conv_stages) && raw_stages > 2)
        raw_stages -= 2;
    while (!fits(raw_stages, conv_stages) && conv_stages > cstep)
        conv_stages -= cstep;
    if (!fits(raw_stages, conv_stages))
        return DSA_ERR_UNSUPPORTED;
    const int smem_bytes =
        static_cast<int>(mx4_smem<D>(R, raw_stages, conv_stages, q_buf_bytes, w_cols, inline_units).total) + 1024;
    if (a.topk.k > 0 &&
        mx4_smem<D>(R, raw_stages, conv_stages, q_buf_bytes, w_cols, inline_units).bar < fused_phase_min_bytes())
        return DSA_ERR_UNSUPPORTED;

    CUtensorMap tm_k;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D / 2), static_cast<uint64_t>(P),
                                  static_cast<uint64_t>(k->num_pages)};
        const uint64_t strides[2] = {static_cast<uint64_t>(k->val_token_stride),
                                     static_cast<uint64_t>(k->val_page_stride)};
        const uint32_t box[3] = {static_cast<uint32_t>(D / 2), static_cast<uint32_t>(P), 1};
        dsa_status st = encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, k->values, dims, strides, box,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != DSA_OK)
            return st;
    }
    Mx4Params p;
    p.sched = a.sched;
    p.context_lens = a.context_lens;
    p.batch = a.batch;
    p.inline_units = inline_units;
    p.block_table = k->block_table;
    p.bt_stride = k->bt_row_stride;
    p.max_pages = k->max_pages_per_seq;
    p.num_pages = k->num_pages;
    p.page_kv = P;
    p.next_n = a.next_n;
    p.ratio = a.ratio;
    p.row_begin = a.row_begin;
    p.row_end = a.row_end;
    p.num_units = a.num_units;
    p.rows_per_unit = G;
    p.q = static_cast<const uint8_t*>(a.q);
    p.q_scales = static_cast<const uint8_t*>(a.q_scales);
    p.q_rows = static_cast<int64_t>(a.batch) * a.next_n * H;
    p.k_scales = static_cast<const uint8_t*>(k->scales);
    p.sc_page_stride = k->sc_page_stride;
    p.weights = a.weights;
    p.logits = a.logits;
    p.logits_stride = a.logits_row_stride;
    p.logits_width = a.logits_width;
    p.status = a.status;
    p.R = R;
    p.raw_stages = raw_stages;
    p.conv_stages = conv_stages;
    p.n_cols = n_cols;
    p.w_cols = w_cols;
    p.acc_cols = acc_cols;
    p.n_acc = n_acc;
    p.n_mma = n_mma;
    p.n_grp = n_grp;
    p.q_buf_bytes = q_buf_bytes;
    p.topk = a.topk;

    auto kern = a.topk.k > 0 ? logits_mxfp4_kernel<D, H, true> : logits_mxfp4_kernel<D, H, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e);
    kern<<<dev.sm_count, kThreads, smem_bytes, stream>>>(tm_k, p);
    return check_launch();
}

template <int D>
dsa_status launch_mx4_d(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    switch (a.num_heads) {
    case 4: return launch_mx4_dh<D, 4>(a, dev, stream);
    case 8: return launch_mx4_dh<D, 8>(a, dev, stream);
    case 16: return launch_mx4_dh<D, 16>(a, dev, stream);
    case 32: return launch_mx4_dh<D, 32>(a, dev, stream);
    case 64: return launch_mx4_dh<D, 64>(a, dev, stream);
    case 128: return launch_mx4_dh<D, 128>(a, dev, stream);
    default: return DSA_ERR_UNSUPPORTED;
    }
}

}  // namespace

dsa_status launch_logits_mxfp4(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    switch (a.k->head_dim) {
    case 64: return launch_mx4_d<64>(a, dev, stream);
    case 128: return launch_mx4_d<128>(a, dev, stream);
    default: return DSA_ERR_UNSUPPORTED;
    }
}

}  // namespace dsa
