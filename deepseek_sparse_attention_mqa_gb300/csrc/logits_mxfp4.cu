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
// path; the ue8m0 block scales stay exact powers of two applied in fp32:
//   warp 0     TMA producer: per 128-token tile one box of packed values and one
//              box of block exponents per physical page into a raw stage ring;
//   warps 6-9  converters: widen a raw tile (one token per thread) into a
//              swizzled K-major e4m3 tile with a byte-permute table, decode the
//              token's block scales to fp32; widen the unit's q rows likewise;
//   warp 1     TMEM allocator + MMA issuer: one M=128 MMA per 32-element block
//              (K = 32) into its own TMEM accumulator, so block scales can be
//              applied per (token, column, block) afterwards;
//   warps 2-9  epilogue (8 warps, two per TMEM lane quarter, splitting the unit's
//              rows): dot = sum_blk 2^(eq+ek-254) * acc_blk, then relu, head
//              weights, store.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "host.h"
#include "logits_common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 448;        // 14 warps: producer, MMA, 8 epilogue, 4 converters
constexpr int kEpiWarps = 8;
constexpr int kFirstConvWarp = 10;
constexpr int kMaxRawStages = 16;
constexpr int kMaxConvStages = 4;
constexpr int kMaxAcc = 4;
constexpr int kPageCache = 512;

struct Mx4Params {
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
    const uint8_t* q;          // packed [R*H][D/2]
    const uint8_t* q_scales;   // [R*H][D/32]
    int64_t q_rows;            // R * H
    const float* weights;
    float* logits;
    int64_t logits_stride;
    int logits_width;
    int32_t* status;
    int n_cols;
    uint32_t acc_cols;         // TMEM columns of one (accumulator, block) slice
    int n_acc;
};

template <int D>
struct Mx4Layout {
    static constexpr int kRawStages = D == 128 ? 8 : kMaxRawStages;
    static constexpr int kConvStages = D == 128 ? 2 : kMaxConvStages;
    static constexpr int kNB = D / 32;                         // blocks (scales) per row
    static constexpr uint32_t kRawK = kTileTokens * D / 2;     // packed bytes per tile
    static constexpr uint32_t kScSlot = 2 * D;                 // bytes per page of exponents (64 x D/32)
    static constexpr uint32_t kConvK = kTileTokens * D;        // e4m3 bytes per tile
    static constexpr uint32_t kLayout = D == 128 ? kLayoutSw128 : kLayoutSw64;
    static constexpr uint32_t kSbo = 8 * D;
};

struct Mx4Smem {
    uint32_t raw_k, raw_sc, conv_k, conv_sc, q, w, sq, pc, bar, misc, total;
};

template <int D>
__host__ __device__ __forceinline__ Mx4Smem mx4_smem(uint32_t q_buf_bytes)
{
    using Lt = Mx4Layout<D>;
    Mx4Smem m;
    m.conv_k = 0;                                                   // 1024-aligned tiles first
    m.q = m.conv_k + Lt::kConvStages * Lt::kConvK;
    m.raw_k = m.q + 2 * q_buf_bytes;
    m.raw_sc = m.raw_k + Lt::kRawStages * Lt::kRawK;
    m.conv_sc = m.raw_sc + Lt::kRawStages * 4 * Lt::kScSlot;      // 4 pages per tile at most
    m.w = m.conv_sc + Lt::kConvStages * kTileTokens * Lt::kNB * 4;
    m.sq = m.w + kEpiWarps * kMaxUnitCols * 4;
    m.pc = m.sq + kEpiWarps * Lt::kNB * kMaxUnitCols * 4;
    m.bar = m.pc + kPageCache * 4;
    m.misc = m.bar + (2 * kMaxRawStages + 2 * kMaxConvStages + 2 * kMaxAcc + 4 + 1) * 8;
    m.total = m.misc + 16;
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
__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8(uint32_t w)
{
    const uint32_t lo_tab = 0x3C383000u, hi_tab = 0x4C484440u;
    const uint32_t lo16 = w & 0xFFFFu, hi16 = w >> 16;
    const uint32_t m0 = __byte_perm(lo_tab, hi_tab, lo16 & 0x7777u);
    const uint32_t s0 = __byte_perm(0u, 0x80808080u, (lo16 & 0x8888u) >> 1);
    const uint32_t m1 = __byte_perm(lo_tab, hi_tab, hi16 & 0x7777u);
    const uint32_t s1 = __byte_perm(0u, 0x80808080u, (hi16 & 0x8888u) >> 1);
    return make_uint2(m0 | s0, m1 | s1);
}

// Widen one packed row (D/2 bytes at src, 16-byte aligned) into row `row` of a
// swizzled K-major e4m3 tile.
template <int D>
__device__ __forceinline__ void widen_row(const uint8_t* src, uint8_t* tile, int row)
{
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {                 // one 16-element chunk = 8 packed bytes
        const uint2 pk = *reinterpret_cast<const uint2*>(src + 8 * c);
        const uint2 a = e2m1x8_to_e4m3x8(pk.x);
        const uint2 b = e2m1x8_to_e4m3x8(pk.y);
        *reinterpret_cast<uint4*>(tile + swizzled_offset(row, c, D)) = make_uint4(a.x, a.y, b.x, b.y);
    }
}

template <int D, int H>
__global__ void __launch_bounds__(kThreads, 1)
logits_mxfp4_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_s,
                    const Mx4Params p)
{
    using Lt = Mx4Layout<D>;
    constexpr int NB = Lt::kNB;
    constexpr int kRawStages = Lt::kRawStages;
    constexpr int kConvStages = Lt::kConvStages;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t q_buf_bytes = ((static_cast<uint32_t>(p.n_cols) * D + 1023u) / 1024u) * 1024u;
    const Mx4Smem mp = mx4_smem<D>(q_buf_bytes);
    uint8_t* sRawK = smem + mp.raw_k;
    uint8_t* sRawS = smem + mp.raw_sc;
    uint8_t* sConvK = smem + mp.conv_k;
    float* sConvS = reinterpret_cast<float*>(smem + mp.conv_sc);
    uint8_t* sQ = smem + mp.q;
    float* sW = reinterpret_cast<float*>(smem + mp.w);
    float* sSq = reinterpret_cast<float*>(smem + mp.sq);
    int* s_pages = reinterpret_cast<int*>(smem + mp.pc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + mp.bar);
    uint64_t* rawf = bars;
    uint64_t* rawe = rawf + kMaxRawStages;
    uint64_t* convf = rawe + kMaxRawStages;
    uint64_t* conve = convf + kMaxConvStages;
    uint64_t* accf = conve + kMaxConvStages;
    uint64_t* acce = accf + kMaxAcc;
    uint64_t* qf = acce + kMaxAcc;
    uint64_t* qe = qf + 2;
    uint64_t* done_bar = qe + 2;
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(smem + mp.misc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + mp.misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(smem_u32(&rawf[s]), 1);
            mbar_init(smem_u32(&rawe[s]), 4);                 // converter warps
        }
        for (int s = 0; s < kConvStages; ++s) {
            mbar_init(smem_u32(&convf[s]), 4);                // converter warps
            mbar_init(smem_u32(&conve[s]), 1 + kEpiWarps);    // MMA commit + epilogue warps
        }
        for (int a = 0; a < kMaxAcc; ++a) {
            mbar_init(smem_u32(&accf[a]), 1);
            mbar_init(smem_u32(&acce[a]), kEpiWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&qf[a]), 4);
            mbar_init(smem_u32(&qe[a]), 1);
        }
        mbar_init(smem_u32(done_bar), 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_s);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), p.n_acc * NB * p.acc_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const WalkParams wp{p.context_lens, p.next_n, p.num_units};
    const int P = p.page_kv;
    const int ppt = kTileTokens / P;

    if (warp == 0) {
        // =========================== TMA producer ===========================
        TileWalk w;
        w.start(wp, units, total_tiles, t0);
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        int pc_unit = -1, pc_lp0 = 0, pc_cnt = 0;
        for (int t = t0; t < t1; ++t) {
            if (*s_abort)
                break;
            w.seek(t);
            const int tt = t - w.ui.tile_begin;
            const int lp_first = tt * ppt;
            if (w.u != pc_unit || lp_first + ppt > pc_lp0 + pc_cnt) {
                const int tiles_here = min(t1, w.ui.tile_end) - w.ui.tile_begin;
                const int lp_vis = (w.ui.vis_max + P - 1) / P;
                const int lp_end = min(tiles_here * ppt, lp_vis);
                const int cnt = min(kPageCache, max(lp_end - lp_first, ppt));
                __syncwarp();
                for (int i = lane; i < cnt; i += 32) {
                    const int lp = lp_first + i;
                    int pg = -1;
                    if (lp < lp_vis && lp < p.max_pages)
                        pg = p.block_table[static_cast<int64_t>(w.ui.seq) * p.bt_stride + lp];
                    s_pages[i] = pg;
                }
                __syncwarp();
                pc_unit = w.u;
                pc_lp0 = lp_first;
                pc_cnt = cnt;
            }
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(smem_u32(&rawe[stage]), phase ^ 1);
                if (ok) {
                    int phys[4];
                    uint32_t bytes = 0;
                    for (int j = 0; j < ppt; ++j) {
                        const int lp = lp_first + j;
                        phys[j] = -1;
                        if (lp * P < w.ui.vis_max) {
                            const int pg = s_pages[lp - pc_lp0];
                            if (pg >= 0 && pg < p.num_pages) {
                                phys[j] = pg;
                                bytes += static_cast<uint32_t>(P) * (D / 2 + NB);
                            } else if (p.status) {
                                atomicOr(p.status, DSA_DEV_BAD_PAGE);
                            }
                        }
                    }
                    const uint32_t fb = smem_u32(&rawf[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    for (int j = 0; j < ppt; ++j) {
                        if (phys[j] < 0)
                            continue;
                        tma_load_3d(smem_u32(sRawK + stage * Lt::kRawK + j * P * (D / 2)), &tm_k, fb, 0, 0, phys[j]);
                        tma_load_2d(smem_u32(sRawS + (stage * 4 + j) * Lt::kScSlot), &tm_s, fb, 0, phys[j]);
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
            if (++stage == kRawStages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (lane == 0) {
            const long long lo = issued > kRawStages ? issued - kRawStages : 0;
            for (long long j = lo; j < issued; ++j)
                mbar_wait(smem_u32(&rawf[j % kRawStages]), static_cast<uint32_t>((j / kRawStages) & 1));
        }
    } else if (warp >= kFirstConvWarp) {
        // =========================== converters =============================
        const int ct = threadIdx.x - kFirstConvWarp * 32;      // 0..127: token of the tile
        TileWalk w;
        w.start(wp, units, total_tiles, t0);
        int rs = 0, cs = 0, ucount = 0;
        uint32_t rph = 0, cph = 0;
        for (int t = t0; t < t1 && !*s_abort; ++t) {
            const bool changed = w.seek(t) || (t == t0);
            if (changed) {
                // widen the unit's q rows into q buffer qb
                const int qb = ucount & 1;
                if (!mbar_wait(smem_u32(&qe[qb]), ((ucount >> 1) & 1) ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                uint8_t* qt = sQ + qb * q_buf_bytes;
                const int64_t r0 = static_cast<int64_t>(w.ui.first_row) * H;
                for (int rr = ct; rr < p.n_cols; rr += 128) {
                    if (r0 + rr < p.q_rows) {
                        widen_row<D>(p.q + (r0 + rr) * (D / 2), qt, rr);
                    } else {
#pragma unroll
                        for (int c = 0; c < D / 16; ++c)
                            *reinterpret_cast<uint4*>(qt + swizzled_offset(rr, c, D)) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&qf[qb]));
                ++ucount;
            }
            if (!mbar_wait(smem_u32(&rawf[rs]), rph) || !mbar_wait(smem_u32(&conve[cs]), cph ^ 1)) {
                *s_abort = 1;
                break;
            }
            // token ct of this tile: page ct / P, row ct % P
            const int j = ct / P, tr = ct % P;
            widen_row<D>(sRawK + rs * Lt::kRawK + ct * (D / 2), sConvK + cs * Lt::kConvK, ct);
            const uint8_t* sc = sRawS + (rs * 4 + j) * Lt::kScSlot + tr * NB;
#pragma unroll
            for (int bk = 0; bk < NB; ++bk)
                sConvS[(cs * kTileTokens + ct) * NB + bk] = ue8m0_to_float(sc[bk]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&rawe[rs]));
                mbar_arrive(smem_u32(&convf[cs]));
            }
            if (++rs == kRawStages) {
                rs = 0;
                rph ^= 1;
            }
            if (++cs == kConvStages) {
                cs = 0;
                cph ^= 1;
            }
        }
    } else if (warp == 1) {
        // =========================== MMA issuer =============================
        if (lane == 0) {
            const uint32_t idesc = make_idesc(0, 0, 0, 128, static_cast<uint32_t>(p.n_cols));
            TileWalk w;
            w.start(wp, units, total_tiles, t0);
            int cs = 0, acc = 0, ucount = 0, qb = 0;
            uint32_t cph = 0, aph = 0;
            for (int t = t0; t < t1 && !*s_abort; ++t) {
                const bool changed = w.seek(t) || (t == t0);
                if (changed) {
                    qb = ucount & 1;
                    if (!mbar_wait(smem_u32(&qf[qb]), (ucount >> 1) & 1)) {
                        *s_abort = 1;
                        break;
                    }
                    ++ucount;
                }
                if (!mbar_wait(smem_u32(&acce[acc]), aph ^ 1) || !mbar_wait(smem_u32(&convf[cs]), cph)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_base = smem_u32(sConvK + cs * Lt::kConvK);
                const uint32_t b_base = smem_u32(sQ + qb * q_buf_bytes);
#pragma unroll
                for (int bk = 0; bk < NB; ++bk) {
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NB + bk) * p.acc_cols;
                    const uint64_t ad = make_smem_desc(a_base + bk * 32, 16, Lt::kSbo, Lt::kLayout);
                    const uint64_t bd = make_smem_desc(b_base + bk * 32, 16, Lt::kSbo, Lt::kLayout);
                    umma_f8f6f4(d_tmem, ad, bd, idesc, 0u);
                }
                umma_commit(smem_u32(&conve[cs]));
                umma_commit(smem_u32(&accf[acc]));
                if ((t + 1 == t1) || (t + 1 >= w.ui.tile_end))
                    umma_commit(smem_u32(&qe[qb]));
                if (++cs == kConvStages) {
                    cs = 0;
                    cph ^= 1;
                }
                if (++acc == p.n_acc) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            umma_commit(smem_u32(done_bar));
            mbar_wait(smem_u32(done_bar), 0);
        }
    } else {
        // =========================== epilogue ===============================
        const int e = warp - 2;                       // 0..7
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const int half = e >> 2;                      // this warp takes unit rows i % 2 == half
        const int tok = quarter * 32 + lane;
        float* wS = sW + e * kMaxUnitCols;
        float* sqS = sSq + e * NB * kMaxUnitCols;
        TileWalk w;
        w.start(wp, units, total_tiles, t0);
        int cs = 0, acc = 0;
        uint32_t cph = 0, aph = 0;
        int L = 0, i0 = 0;
        for (int t = t0; t < t1 && !__any_sync(0xffffffffu, *s_abort); ++t) {
            const bool changed = w.seek(t) || (t == t0);
            if (changed) {
                __syncwarp();
                const int nvalid = w.ui.nrows * H;
                const int64_t c0 = static_cast<int64_t>(w.ui.first_row) * H;
                for (int c = lane; c < kMaxUnitCols; c += 32) {
                    wS[c] = c < nvalid ? p.weights[c0 + c] : 0.f;
#pragma unroll
                    for (int bk = 0; bk < NB; ++bk)
                        sqS[bk * kMaxUnitCols + c] = c < nvalid ? ue8m0_to_float(p.q_scales[(c0 + c) * NB + bk]) : 0.f;
                }
                __syncwarp();
                L = max(0, p.context_lens[w.ui.seq]);
                i0 = w.ui.first_row - w.ui.seq * p.next_n;
                if (e == 0 && lane == 0 && p.status &&
                    visible_len(L, p.next_n, i0 + w.ui.nrows - 1) > p.logits_width)
                    atomicOr(p.status, DSA_DEV_WIDTH);
            }
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&convf[cs]), cph) && mbar_wait(smem_u32(&accf[acc]), aph))) {
                *s_abort = 1;
                break;
            }
            tc_fence_after_sync();
            float sk[NB];
#pragma unroll
            for (int bk = 0; bk < NB; ++bk)
                sk[bk] = sConvS[(cs * kTileTokens + tok) * NB + bk];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&conve[cs]));
            const int s = (t - w.ui.tile_begin) * kTileTokens + tok;
            const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            // rows of the unit handled by this warp: i = half, half + 2, ...
            for (int i = half; i < w.ui.nrows; i += 2) {
                float rowsum = 0.f;
                const int c_lo = i * H, c_hi = (i + 1) * H;
                // 32-column chunks aligned within the accumulator slice (a row of
                // H < 32 heads lies inside one chunk)
                for (int cb = c_lo & ~31; cb < c_hi; cb += 32) {
                    float dot[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        dot[j] = 0.f;
#pragma unroll
                    for (int bk = 0; bk < NB; ++bk) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(t_acc + static_cast<uint32_t>(acc * NB + bk) * p.acc_cols + cb, r);
                        tmem_ld_wait();
                        const float* sq = sqS + bk * kMaxUnitCols + cb;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            dot[j] = fmaf(sq[j] * sk[bk], __uint_as_float(r[j]), dot[j]);
                    }
                    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (cb + j >= c_lo && cb + j < c_hi)
                            part[j & 3] = fmaf(wS[cb + j], fmaxf(dot[j], 0.f), part[j & 3]);
                    rowsum += (part[0] + part[1]) + (part[2] + part[3]);
                }
                const int vis = min(visible_len(L, p.next_n, i0 + i), p.logits_width);
                if (s < vis)
                    p.logits[static_cast<int64_t>(w.ui.first_row + i - p.row_begin) * p.logits_stride + s] = rowsum;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&acce[acc]));
            if (++cs == kConvStages) {
                cs = 0;
                cph ^= 1;
            }
            if (++acc == p.n_acc) {
                acc = 0;
                aph ^= 1;
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
        tmem_dealloc(tmem_base, p.n_acc * NB * p.acc_cols);
}

template <int D, int H>
dsa_status launch_mx4_dh(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    using Lt = Mx4Layout<D>;
    const dsa_paged_cache* k = a.k;
    const int P = k->page_kv;
    const int G = a.rows_per_unit;
    const int n_cols = ((G * H + 15) / 16) * 16;
    uint32_t acc_cols = 32;
    while (acc_cols < static_cast<uint32_t>(n_cols))
        acc_cols <<= 1;
    // n_acc accumulators x NB blocks x acc_cols columns within 512, a power of two
    int n_acc = kMaxAcc;
    while (n_acc > 1 && static_cast<uint32_t>(n_acc) * Lt::kNB * acc_cols > 512u)
        n_acc >>= 1;
    if (static_cast<uint32_t>(n_acc) * Lt::kNB * acc_cols > 512u)
        return DSA_ERR_UNSUPPORTED;
    if (P * Lt::kNB > static_cast<int>(Lt::kScSlot))
        return DSA_ERR_UNSUPPORTED;
    const uint32_t q_buf_bytes = ((static_cast<uint32_t>(n_cols) * D + 1023u) / 1024u) * 1024u;
    const Mx4Smem mp = mx4_smem<D>(q_buf_bytes);
    const int smem_bytes = static_cast<int>(mp.total) + 1024;
    if (smem_bytes > std::min(dev.max_smem_optin, 227 * 1024))
        return DSA_ERR_UNSUPPORTED;

    CUtensorMap tm_k, tm_s;
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
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(P * Lt::kNB), static_cast<uint64_t>(k->num_pages)};
        const uint64_t strides[1] = {static_cast<uint64_t>(k->sc_page_stride)};
        const uint32_t box[2] = {static_cast<uint32_t>(P * Lt::kNB), 1};
        dsa_status st = encode_tiled(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k->scales, dims, strides, box,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != DSA_OK)
            return st;
    }
    Mx4Params p;
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
    p.q = static_cast<const uint8_t*>(a.q);
    p.q_scales = static_cast<const uint8_t*>(a.q_scales);
    p.q_rows = static_cast<int64_t>(a.batch) * a.next_n * H;
    p.weights = a.weights;
    p.logits = a.logits;
    p.logits_stride = a.logits_row_stride;
    p.logits_width = a.logits_width;
    p.status = a.status;
    p.n_cols = n_cols;
    p.acc_cols = acc_cols;
    p.n_acc = n_acc;

    auto kern = logits_mxfp4_kernel<D, H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e);
    kern<<<dev.sm_count, kThreads, smem_bytes, stream>>>(tm_k, tm_s, p);
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
