// mla_tc.cu -- sparse MLA decode on the tcgen05 tensor cores (DeepSeek latent
// attention shapes: up to 128 query heads, q/k dim 512 or 576, v dim 512, FP8
// e4m3 latent cache with one fp32 scale per token).
//
// "Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels" (flashinfer #3269): decode
// attention of each query row over the latent tokens its top-k selected, with
// bf16 output and an LSE output; the pages give precompiled kernels and a
// multi-CTA reduction for it, neither of which is used here.
//
// GB300 design: one CLUSTER of two CTAs per query row.  The output O
// (128 heads x 512 fp32) fills a whole TMEM, so it is split by value dims:
// CTA c owns latent dims [256 c, 256 c + 256) and, at d_qk 576, half of the
// rope dims, [512 + 32 c, 544 + 32 c), so both do equal work; each keeps its
// part of Q resident (f16, times a per-head power of two that fits it to f16
// range exactly: the 256 value dims in TMEM as the A operand of the QK MMA,
// the rope dims in a swizzled K-major shared-memory tile), gathers and widens
// its part of the selected latent rows (FP8 -> f16, exact) and computes a PARTIAL score
// S_c = Q_c K_c^T on the tensor cores.  The two partials are exchanged through
// distributed shared memory, so both CTAs hold the same S = S_0 + S_1 (identical
// arithmetic, hence identical softmax decisions) and each accumulates its half
// of O = P V in TMEM, where V is the first 256 dims of its own latent slice.
//
//   warps 0-3, 9-12  softmax, two threads per head (TMEM lane = head): warps
//              0-3 take tokens 0-31 of each block, warps 9-12 tokens 32-63.
//              Each warp sends its partial scores to the same warp of the peer
//              CTA with one bulk shared-memory copy (completing on that warp's
//              mbarrier), adds the peer's, scales and masks each token pair with
//              one packed FMA (token scale * softmax scale * log2 e, and a -inf
//              bias for empty slots) and keeps an online max / sum in base 2
//              (packed fp32 pairs, hardware exp2); the two threads of a head combine their
//              block maxima through shared memory and a two-thread mbarrier.
//              The running max is refreshed lazily (O in TMEM is rescaled only
//              when the max grows by more than 2^8).  P is written as f16
//              (token scale folded in for V; f16 rather than bf16 keeps its
//              rounding at 2^-12); at the end O is normalised and stored as
//              bf16 out / fp32 lse.
//   warps 4-7  gather, three latent tiles in flight: per 64-token block, look
//              up each selected token through the block table (two blocks
//              ahead), load its FP8 slice (the
//              next block's loads are issued before this block's widening
//              stores), widen to f16 into a 128B-swizzled K-major tile (zeros
//              for unused slots).
//   warp 8     TMEM allocator + MMA issuer: S = Q K^T (M=128, N=64) and
//              O += P V (M=128, N=256, V read MN-major from the same tile),
//              each issued as soon as its inputs are ready.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kNT = 64;                 // selected tokens per block
constexpr int kMaxChunks = 5;           // 64-dim tile chunks per CTA (4 value chunks + a half-used rope chunk)
constexpr int kVChunks = 4;             // 256 value dims per CTA
constexpr int kQChunkBytes = 128 * 128; // 128 heads x 64 f16
constexpr int kLChunkBytes = kNT * 128; // 64 tokens x 64 f16
constexpr int kThreads = 416;           // 13 warps
constexpr int kConvWarp0 = 4;           // gather warps 4-7
constexpr int kMmaWarp = 8;
constexpr int kSoftWarp1 = 9;           // softmax warps 0-3 (tokens 0-31) and 9-12 (tokens 32-63)
constexpr uint32_t kTmemCols = 512;     // S[2] at columns 0 / 64, Q (value dims, f16 pairs) at 128, O at 256
constexpr uint32_t kQCol = 128;
constexpr int kLatBufs = 3;             // latent tiles (with their per-token scales, multipliers and biases) in flight
constexpr float kRescaleLog2 = 8.f;     // refresh the running max only past 2^8
constexpr int kMaxSeg = 18;             // 16-byte FP8 segments per token and CTA (256 + 32 dims)
constexpr int kGatherItems = (16 * kMaxSeg + 31) / 32;      // 16-byte segments per gather lane

struct MlaParams {
    const __nv_bfloat16* q;
    int num_heads;
    int d_qk;
    float scale_log2;                   // softmax_scale * log2(e)
    const uint8_t* vals;
    int64_t vps, vts;
    const uint8_t* scs;
    int64_t sps, sts;
    const int32_t* bt;
    int64_t bt_stride;
    int max_pages;
    int page_kv;
    int num_pages;
    const int32_t* seq_of_row;
    int next_n;
    const int32_t* idx;
    int64_t idx_stride;
    int k;
    __nv_bfloat16* out;
    float* lse;
    int32_t* status;
    // per-row top-k lengths, the sliding-window cache and varlen rows (null: none)
    const int32_t* topk_lens;
    const uint8_t* wvals;
    int64_t wvps, wvts;
    const uint8_t* wscs;
    int64_t wsps, wsts;
    const int32_t* wbt;
    int64_t wbt_stride;
    int wmax_pages;
    int wpage_kv;
    int wnum_pages;
    int window;
    const int32_t* seq_lens;
    const int32_t* cum_q;
    int batch;
};

struct MlaSmem {
    uint32_t q, lat, p, x, xs, scale, mult, bias, qexp, red, bar, misc, total;
};

__host__ __device__ constexpr MlaSmem mla_smem()
{
    MlaSmem m{};
    m.q = 0;
    m.lat = m.q + kQChunkBytes;                      // the rope chunk of Q (value dims are in TMEM)
    m.p = m.lat + kLatBufs * kMaxChunks * kLChunkBytes;  // (P lives in TMEM, in its block's S columns)
    m.x = m.p;
    m.xs = m.x + 128 * kNT * 4;                      // this CTA's partial scores, staged for the peer
    m.scale = m.xs + 128 * kNT * 4;
    m.mult = m.scale + kLatBufs * kNT * 4;          // per token: scale * softmax scale * log2(e), 0 if none
    m.bias = m.mult + kLatBufs * kNT * 4;            // per token: 0, or -inf for a slot with no token
    m.qexp = m.bias + kLatBufs * kNT * 4;
    m.red = m.qexp + 128 * 4;
    m.bar = m.red + 2 * 2 * 128 * 4;
    m.misc = m.bar + 40 * 8;
    m.total = m.misc + 16;
    return m;
}

// tcgen05.mma kind::f16 with the A operand in tensor memory (lane = row of A,
// two 16-bit K elements per 32-bit column; one K step of 16 = 8 columns).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 e4m3 bytes -> 16 f16 (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x16_to_f16x16(const uint4 v, uint4& lo, uint4& hi)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hh)) & 0xFFFFu);
            const __half2_raw h2r = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            o[2 * i + hh] = static_cast<uint32_t>(h2r.x) | (static_cast<uint32_t>(h2r.y) << 16);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 2^e as fp32 for |e| <= 126 (exact).
__device__ __forceinline__ float exp2_int(int e)
{
    return __int_as_float((127 + e) << 23);
}

// kDual: per-row top-k lengths, the sliding-window cache and cumulative query
// lengths; without it the kernel reads the index lists alone (the gather keeps
// fewer values live).
template <bool kDual>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const MlaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr MlaSmem mp = mla_smem();
    uint8_t* sQ = smem + mp.q;
    uint8_t* sLat = smem + mp.lat;
    uint8_t* sX = smem + mp.x;
    uint8_t* sXs = smem + mp.xs;
    float* sScale = reinterpret_cast<float*>(smem + mp.scale);
    float* sMult = reinterpret_cast<float*>(smem + mp.mult);
    float* sBias = reinterpret_cast<float*>(smem + mp.bias);
    int* sQexp = reinterpret_cast<int*>(smem + mp.qexp);       // per-head power-of-two Q scale
    float* sMax = reinterpret_cast<float*>(smem + mp.red);        // [2][128] block max per half
    float* sSum = sMax + 2 * 128;                                  // [2][128] final sum per half
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + mp.bar);
    uint64_t* q_full = bars + 0;
    uint64_t* lat_full = bars + 1;   // [kLatBufs]
    uint64_t* lat_empty = bars + 4;  // [kLatBufs]
    uint64_t* s_full = bars + 7;     // [2]
    uint64_t* s_empty = bars + 9;    // [2]
    uint64_t* xw_full = bars + 24;   // [8] per softmax warp: the peer's partial scores arrived in sX
    uint64_t* xw_free = bars + 32;   // [8] per softmax warp: the peer consumed what this warp sent
    // [2] per S/P buffer: the 8 softmax warps wrote P of the buffer's block.  One
    // barrier per buffer, because a warp may write P(j + 1) before a warp of
    // another lane quarter has written P(j); P(j + 2) cannot come before PV(j)
    // has completed, so a phase never mixes two blocks' arrivals.
    uint64_t* p_full = bars + 11;
    uint64_t* q_stage = bars + 13;   // the Q slice staged in shared memory
    uint64_t* p_empty = bars + 14;
    uint64_t* o_done = bars + 15;
    uint64_t* pair_bar = bars + 16;  // [4] the two softmax warps of a lane quarter
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(smem + mp.misc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + mp.misc + 4);

    // launched as a programmatic dependent of the previous kernel of the stream
    // (the top-k): nothing is read before this wait, so only the launch latency
    // overlaps its end
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t peer = crank ^ 1u;
    const int row = blockIdx.y;
    const MlaRowSeq rs = kDual ? mla_row_seq(row, p.cum_q, p.batch, p.seq_of_row, p.next_n)
                               : MlaRowSeq{p.seq_of_row ? p.seq_of_row[row] : row / p.next_n, 0, 1};
    const int seq = rs.seq;
    // this row's token slots: the first kr entries of its index list, then the
    // w window positions [win0, win0 + w) of the window cache
    int kr = p.k, w = 0, win0 = 0;
    if (!kDual) {
    } else if (seq < 0) {
        kr = 0;                                  // a row outside every sequence: no key
        if (threadIdx.x == 0 && cluster_ctarank() == 0 && p.status)
            atomicOr(p.status, DSA_DEV_BAD_INDEX);
    } else {
        if (p.topk_lens)
            kr = min(max(p.topk_lens[row], 0), p.k);
        if (p.wvals) {
            const int vis = visible_len(max(p.seq_lens[seq], 0), rs.q_len, rs.i);
            w = min(p.window, vis);
            win0 = vis - w;
        }
    }
    const int nslots = kr + w;
    // Latent dims of this CTA: its value dims [256 c, 256 c + 256) (tile chunks
    // 0-3, also V for its half of O) and, at d_qk 576, half of the rope dims,
    // [512 + 32 c, 544 + 32 c) (the first half of tile chunk 4), so that both
    // CTAs gather and multiply 288 dims per token and neither waits for the
    // other at the score exchange.
    const bool rope = p.d_qk == 576;
    const int nchunk = rope ? kVChunks + 1 : kVChunks;
    const int nseg = rope ? kMaxSeg : 16;            // 16-byte FP8 segments per token
    // latent dim of this CTA's 16-dim segment sg (FP8 byte offset in the row)
    auto seg_dim = [&](int sg) -> int {
        return sg < 16 ? static_cast<int>(crank) * 256 + sg * 16 : 512 + static_cast<int>(crank) * 32 + (sg - 16) * 16;
    };
    const int nblk = (nslots + kNT - 1) / kNT;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(q_full), 4);
        mbar_init(smem_u32(q_stage), 1);
        for (int i = 0; i < kLatBufs; ++i) {
            mbar_init(smem_u32(&lat_full[i]), 4);
            mbar_init(smem_u32(&lat_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_empty[i]), 1);   // PV of the block that used the buffer (it holds P)
            mbar_init(smem_u32(&p_full[i]), 8);
        }
        for (int i = 0; i < 8; ++i) {
            mbar_init(smem_u32(&xw_full[i]), 1);    // local expect_tx + the peer warp's bulk copy bytes
            mbar_init(smem_u32(&xw_free[i]), 1);    // the peer warp's remote arrive
        }
        mbar_init(smem_u32(p_empty), 1);
        mbar_init(smem_u32(o_done), 1);
        for (int i = 0; i < 4; ++i)
            mbar_init(smem_u32(&pair_bar[i]), 2);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();              // the peer's barriers are initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *s_tmem;

    if (warp >= kConvWarp0 && warp < kMmaWarp) {
        // ================================ gather ================================
        const int ct = threadIdx.x - kConvWarp0 * 32;   // 0..127
        // Q slice -> f16.  Thread ct owns head ct: Q is scaled by 2^e, e chosen
        // per head from this CTA's slice so that max|q| 2^e lies in [2^14, 2^15)
        // -- exact, and inside f16 range whatever the bf16 magnitudes; the
        // partial scores are scaled back by 2^-e in fp32.  The slice is first
        // staged in shared memory (the latent tiles are not in use yet) by five
        // TMA boxes of 128 heads x 64 dims, 128B-swizzled: its four 64-dim value
        // chunks and the rope chunk (dims 512-575, of which this CTA takes 32),
        // so that one thread per head reads its 16-byte units without bank
        // conflicts.  Read directly from global memory, each warp load touched
        // 32 rows 1152 B apart and the loads serialised in the load/store unit.
        const uint8_t* qst = sLat;
        const int nunit = 2 * nseg;
        if (warp == kConvWarp0 && lane == 0) {
            const int nbox = rope ? 5 : 4;
            mbar_arrive_expect_tx(smem_u32(q_stage), static_cast<uint32_t>(nbox * 128 * 128));
            for (int b = 0; b < nbox; ++b)
                tma_load_2d(smem_u32(qst + b * 128 * 128), &tm_q, smem_u32(q_stage),
                            b < 4 ? static_cast<int>(crank) * 256 + 64 * b : 512, row * p.num_heads);
        }

        const int32_t* irow = p.idx + static_cast<int64_t>(row) * p.idx_stride;
        const int gw = warp - kConvWarp0;               // this warp gathers tokens [16 gw, 16 gw + 16) of a block
        // Lane l < 16 owns token gw * 16 + l of every block.  Finding a token's
        // latent row takes three dependent global loads (index -> block table ->
        // row and scale), so they are software-pipelined across iterations: while
        // block j is stored, the latent loads of block j + 1 fly, block j + 2's
        // row address is formed from the block-table entry loaded one iteration
        // earlier, block j + 3's block-table entry is loaded and block j + 4's
        // index.  Each load thus has a whole iteration to land.
        auto tok_of = [&](int jb) -> int { return jb * kNT + gw * 16 + lane; };
        // a slot's token: an index of the sparse cache, a window position tagged
        // with kSwaTag, or -1 (no token: padding or past the row's slots)
        auto load_idx = [&](int jb) -> int {
            if (lane >= 16 || jb >= nblk)
                return -1;
            const int t = tok_of(jb);
            if (!kDual)
                return t < p.k ? irow[t] : -1;
            if (t < kr)
                return irow[t];
            return t < nslots ? ((win0 + t - kr) | kSwaTag) : -1;
        };
        auto load_page = [&](int sidx) -> int {    // block-table entry of a token (-1 if none)
            if (sidx < 0)
                return -1;
            if (kDual && (sidx & kSwaTag)) {
                const int lp = (sidx & ~kSwaTag) / p.wpage_kv;
                return lp < p.wmax_pages ? p.wbt[static_cast<int64_t>(seq) * p.wbt_stride + lp] : -1;
            }
            const int lp = sidx / p.page_kv;
            return lp < p.max_pages ? p.bt[static_cast<int64_t>(seq) * p.bt_stride + lp] : -1;
        };
        // row address of a token from its index and page: the latent row's and
        // its scale's global addresses, or valid = 0 (a selected token with no
        // valid page is reported and contributes nothing)
        auto address = [&](int sidx, int pg, int64_t& off, int64_t& soff, int& valid) {
            off = 0;
            soff = 0;
            valid = 0;
            if (sidx < 0)
                return;
            const bool swa = kDual && (sidx & kSwaTag) != 0;
            const int pos = kDual ? (sidx & ~kSwaTag) : sidx;
            const int P = swa ? p.wpage_kv : p.page_kv;
            if (pg >= 0 && pg < (swa ? p.wnum_pages : p.num_pages)) {
                const uint8_t* v = swa ? p.wvals + pg * p.wvps + (pos % P) * p.wvts
                                       : p.vals + pg * p.vps + (pos % P) * p.vts;
                const uint8_t* sc = swa ? p.wscs + pg * p.wsps + (pos % P) * p.wsts
                                        : p.scs + pg * p.sps + (pos % P) * p.sts;
                off = static_cast<int64_t>(reinterpret_cast<uintptr_t>(v));
                soff = static_cast<int64_t>(reinterpret_cast<uintptr_t>(sc));
                valid = 1;
            } else if (p.status) {
                atomicOr(p.status, DSA_DEV_BAD_INDEX);
            }
        };
        auto load_scale = [&](int64_t soff, int valid) -> float {
            return valid ? *reinterpret_cast<const float*>(static_cast<uintptr_t>(soff)) : 0.f;
        };
        auto issue_loads = [&](uint4 (&raw)[kGatherItems], int64_t off, int valid) {
#pragma unroll
            for (int i = 0; i < kGatherItems; ++i) {
                const int flat = i * 32 + lane;
                const int tl = flat / nseg, seg = flat % nseg;
                const int64_t o = __shfl_sync(0xffffffffu, off, tl & 15);
                const int v = __shfl_sync(0xffffffffu, valid, tl & 15);
                raw[i] = make_uint4(0, 0, 0, 0);
                if (flat < 16 * nseg && v)
                    raw[i] = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(static_cast<uintptr_t>(o)) +
                                                             seg_dim(seg));
            }
        };
        // prologue: indices of blocks 0-3, pages of blocks 0-2, addresses of 0-1
        int s0 = load_idx(0), s1 = load_idx(1), s2 = load_idx(2), s3 = load_idx(3);
        const int pg0 = load_page(s0), pg1 = load_page(s1);
        int pg2 = load_page(s2);
        // (the index and block-table loads above fly while Q is prepared)
        bool q_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(q_stage), 0));
        if (!q_ok)
            *s_abort = 1;
        {
            const int h = ct;
            const bool hv = q_ok && h < p.num_heads;
            auto unit = [&](int u) -> uint4 {
                // value unit u < 32: box u / 8, 16-byte unit u % 8 of head h's 128 B row;
                // rope unit u - 32: box 4, unit 4 crank + u - 32
                const uint32_t off = u < 32 ? (u >> 3) * 16384u + swizzled_offset(h, u & 7, 128)
                                            : 4u * 16384u + swizzled_offset(h, crank * 4 + (u - 32), 128);
                return hv ? *reinterpret_cast<const uint4*>(qst + off) : make_uint4(0, 0, 0, 0);
            };
            // max |q| of the slice: for non-negative bf16 values the order of the bit
            // patterns as unsigned 16-bit integers is the order of the values, so
            // the sign bits are masked off and two values are compared per
            // packed integer max
            uint32_t m2 = 0;
#pragma unroll 4
            for (int u = 0; u < nunit; ++u) {
                const uint4 v = unit(u);
                m2 = __vmaxu2(m2, __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
                m2 = __vmaxu2(m2, __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
            }
            const float amax = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
            int e = 0;
            if (amax > 0.f && amax <= 3.0e38f) {
                int ex;
                frexpf(amax, &ex);                          // amax in [2^(ex-1), 2^ex)
                e = max(-100, min(100, 15 - ex));
            }
            sQexp[h] = e;
            const float sc = exp2_int(e);
            const uint64_t sc2 = pack_f32x2(sc, sc);
            auto conv = [&](int u) -> uint4 {              // 8 dims of unit u, f16 x 2^e
                const uint4 v = unit(u);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                uint32_t r4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // bf16 -> fp32 is a 16-bit shift; times 2^e (exact), then f16
                    const float2 f = unpack_f32x2(mul_f32x2(
                        pack_f32x2(__uint_as_float(w4[i] << 16), __uint_as_float(w4[i] & 0xFFFF0000u)), sc2));
                    const __half2 hf = __floats2half2_rn(f.x, f.y);
                    r4[i] = *reinterpret_cast<const uint32_t*>(&hf);
                }
                return make_uint4(r4[0], r4[1], r4[2], r4[3]);
            };
            // the 256 value dims go to TMEM lane h (this warp's lane quarter),
            // columns [kQCol, kQCol + 128): 32 columns (8 units) per store
            const uint32_t q_lane = static_cast<uint32_t>((warp & 3) * 32) << 16;
#pragma unroll 1
            for (int r = 0; r < 4; ++r) {
                uint32_t wv[32];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const uint4 o = conv(8 * r + b);
                    wv[4 * b] = o.x;
                    wv[4 * b + 1] = o.y;
                    wv[4 * b + 2] = o.z;
                    wv[4 * b + 3] = o.w;
                }
                tmem_st_32x32b_x32(tmem_base + q_lane + kQCol + 32 * r, wv);
            }
            tmem_st_wait();
            // the rope dims (d_qk 576) go to the shared-memory chunk
            for (int u = 32; u < nunit; ++u)
                *reinterpret_cast<uint4*>(sQ + swizzled_offset(h, u - 32, 128)) = conv(u);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(q_full));
        // all four gather warps read staged Q rows from the latent tiles: none
        // writes a tile before all are done (named barrier 1, the 128 gather threads)
        named_bar_sync(1, 128);
        int64_t off0, soff0, off1, soff1;
        int valid0, valid1;
        address(s0, pg0, off0, soff0, valid0);
        address(s1, pg1, off1, soff1, valid1);
        uint4 raw[kGatherItems];
        issue_loads(raw, off0, valid0);
        float scale0 = load_scale(soff0, valid0);
        for (int j = 0; j < nblk && !__any_sync(0xffffffffu, *s_abort); ++j) {
            const int st = j % kLatBufs;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&lat_empty[st]), ((j / kLatBufs) & 1) ^ 1))) {
                *s_abort = 1;
                break;
            }
            uint8_t* tile = sLat + st * (kMaxChunks * kLChunkBytes);
#pragma unroll
            for (int i = 0; i < kGatherItems; ++i) {
                const int flat = i * 32 + lane;
                if (flat >= 16 * nseg)
                    continue;
                const int tl = flat / nseg, seg = flat % nseg;
                uint4 lo, hi;
                e4m3x16_to_f16x16(raw[i], lo, hi);       // zero bytes (unused slot) -> zeros
                uint8_t* chunk = tile + (seg >> 2) * kLChunkBytes;
                const int un = (seg & 3) * 2;
                *reinterpret_cast<uint4*>(chunk + swizzled_offset(gw * 16 + tl, un, 128)) = lo;
                *reinterpret_cast<uint4*>(chunk + swizzled_offset(gw * 16 + tl, un + 1, 128)) = hi;
            }
            if (lane < 16) {
                sScale[st * kNT + gw * 16 + lane] = scale0;
                sMult[st * kNT + gw * 16 + lane] = valid0 ? scale0 * p.scale_log2 : 0.f;
                sBias[st * kNT + gw * 16 + lane] = valid0 ? 0.f : -INFINITY;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&lat_full[st]));
            // block j + 1: latent loads and its scale (zeros past the end)
            issue_loads(raw, off1, valid1);
            const float scale1 = load_scale(soff1, valid1);
            // block j + 2: row address from the page loaded last iteration
            int64_t off2, soff2;
            int valid2;
            address(s2, pg2, off2, soff2, valid2);
            // block j + 3: its page; block j + 4: its index
            const int pg3 = load_page(s3);
            const int s4 = load_idx(j + 4);
            valid0 = valid1;
            scale0 = scale1;
            off1 = off2;
            soff1 = soff2;
            valid1 = valid2;
            s2 = s3;
            pg2 = pg3;
            s3 = s4;
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA ===================================
        if (lane == 0) {
            const uint32_t idesc_qk = make_idesc(0, 0, 0, 128, kNT);     // f16 x f16 -> f32
            const uint32_t idesc_pv = make_idesc(0, 0, 1, 128, 256);
            bool ok = mbar_wait(smem_u32(q_full), 0);
            // Two independent streams share this thread: S(j) = Q K_j^T once block j
            // is gathered (and the S buffer is free), and O += P_j V_j once the
            // softmax has written P_j.  Whichever is ready is issued, so a PV never
            // waits behind the gather of a later block (which itself waits for
            // that PV to free its latent buffer).
            auto issue_qk = [&](int j) {
                const int st = j & 1;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + static_cast<uint32_t>(st * kNT);
                const uint32_t qa = smem_u32(sQ);
                const uint32_t kb = smem_u32(sLat + (j % kLatBufs) * (kMaxChunks * kLChunkBytes));
                for (int ch = 0; ch < nchunk; ++ch) {
                    const int nks = ch < kVChunks ? 4 : 2;       // the rope chunk holds 32 dims
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        if (ks >= nks)
                            break;
                        const uint64_t bd = make_smem_desc(kb + ch * kLChunkBytes + ks * 32, 16, 1024, kLayoutSw128);
                        if (ch < kVChunks) {
                            // value dims: A = Q from TMEM (16 K elements = 8 columns per step)
                            umma_f16_ts(d, tmem_base + kQCol + ch * 32 + ks * 8, bd, idesc_qk, (ch | ks) != 0 ? 1u : 0u);
                        } else {
                            const uint64_t ad = make_smem_desc(qa + ks * 32, 16, 1024, kLayoutSw128);
                            umma_f16(d, ad, bd, idesc_qk, 1u);
                        }
                    }
                }
                umma_commit(smem_u32(&s_full[st]));
            };
            auto issue_pv = [&](int j) {
                tc_fence_after_sync();
                // O[:, v] += P[:, t] V[t, v]: A = P from TMEM (lane = head, the f16
                // token pairs the softmax wrote over this block's S columns, 8
                // columns per 16-token step), B = V read MN-major from the latent
                // tile (64-dim blocks 8 KB apart = LBO, 8-token groups 1 KB apart = SBO)
                const uint32_t d = tmem_base + 256;
                const uint32_t pa = tmem_base + static_cast<uint32_t>((j & 1) * kNT);
                const uint32_t vb = smem_u32(sLat + (j % kLatBufs) * (kMaxChunks * kLChunkBytes));
#pragma unroll
                for (int ks = 0; ks < kNT / 16; ++ks) {
                    const uint64_t bd = make_smem_desc(vb + ks * 2048, kLChunkBytes, 1024, kLayoutSw128);
                    umma_f16_ts(d, pa + ks * 8, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(p_empty));
                umma_commit(smem_u32(&lat_empty[j % kLatBufs]));
                umma_commit(smem_u32(&s_empty[j & 1]));   // the S/P buffer is free for QK(j + 2)
            };
            int jq = 0, jp = 0;                         // next QK / PV block to issue
            uint64_t t_idle = 0;
            while (ok && jp < nblk && !*s_abort) {
                bool progress = false;
                // QK(jq): its latent block is gathered and S buffer jq & 1 was read
                if (jq < nblk && mbar_test_wait(smem_u32(&lat_full[jq % kLatBufs]), (jq / kLatBufs) & 1) &&
                    mbar_test_wait(smem_u32(&s_empty[jq & 1]), ((jq >> 1) & 1) ^ 1)) {
                    issue_qk(jq++);
                    progress = true;
                }
                // PV(jp): P_jp is written (S(jp) was issued before, so jp < jq)
                if (jp < jq && mbar_test_wait(smem_u32(&p_full[jp & 1]), (jp >> 1) & 1)) {
                    issue_pv(jp++);
                    progress = true;
                }
                if (progress) {
                    t_idle = 0;
                    continue;
                }
                if (t_idle == 0) {
                    t_idle = global_timer_ns();
                } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
                    ok = false;
                }
            }
            if (!ok)
                *s_abort = 1;
            umma_commit(smem_u32(o_done));
            mbar_wait(smem_u32(o_done), 0);
        }
    } else {
        // ================================ softmax ===============================
        // Two threads per head (= TMEM lane): warps 0-3 take tokens [0, 32) of
        // every block, warps 9-12 tokens [32, 64); the pair agrees on the block
        // max through shared memory and a named barrier, and keeps the running
        // max in lockstep (both see the same sequence of block maxima).
        const int quarter = warp & 3;
        const int half = warp >= kSoftWarp1 ? 1 : 0;
        const int h = quarter * 32 + lane;                // head = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int tcol = half * 32;                       // this thread's tokens within a block
        // the two warps of this lane quarter meet on pair_bar[quarter] (bounded
        // waits, so a warp that gives up cannot strand its partner)
        uint32_t pair_uses = 0;
        auto pair_sync = [&]() -> bool {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&pair_bar[quarter]));
            const bool r = __all_sync(0xffffffffu, mbar_wait(smem_u32(&pair_bar[quarter]), pair_uses & 1));
            tc_fence_after_sync();
            ++pair_uses;
            return r;
        };
        // Score exchange, per softmax warp: this warp's 32 threads stage their 32
        // partial scores (128 B each, 16-byte units XOR-swizzled by lane) in its
        // 4 KB slice of sXs, and one lane copies the slice with a single bulk
        // shared-memory copy into the same slice of the peer's sX, where the
        // peer's warp of the same (quarter, half) -- the same heads and tokens --
        // reads it; the copy completes on that warp's own mbarrier.
        const int widx = half * 4 + quarter;
        uint8_t* stage_row = sXs + widx * 4096 + lane * 128;
        const uint8_t* recv_row = sX + widx * 4096 + lane * 128;
        const uint32_t peer_slice = mapa_shared(smem_u32(sX + widx * 4096), peer);
        const uint32_t peer_full = mapa_shared(smem_u32(&xw_full[widx]), peer);
        const uint32_t peer_free = mapa_shared(smem_u32(&xw_free[widx]), peer);
        float m_run = -INFINITY, l_run = 0.f;
        // this head's Q was stored times 2^e; partial scores are scaled back (exact)
        bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(q_full), 0));
        const float qback = exp2_int(-sQexp[h]);
        for (int j = 0; j < nblk && ok; ++j) {
            const int sb = j & 1;
            const uint32_t ph = (j >> 1) & 1;
            // every wait outcome is made warp-uniform: the tcgen05 loads and stores
            // below are .sync.aligned and must be executed by all 32 lanes together
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[sb]), ph))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            uint32_t ra[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + sb * kNT + tcol, ra);
            tmem_ld_wait();
            // this CTA's partial scores as token pairs, scaled back by 2^-e (exact)
            uint64_t sc2[16];
            const uint64_t qb2 = pack_f32x2(qback, qback);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                sc2[i] = mul_f32x2(pack_f32x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])), qb2);

            // ---- exchange partial scores with the peer CTA (one bulk copy per warp)
            if (lane == 0)
                mbar_arrive_expect_tx(smem_u32(&xw_full[widx]), 4096u);
            // the peer has consumed this warp's previous copy (so it has landed and
            // this warp's staging slice was read)
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&xw_free[widx]), (j & 1) ^ 1))) {
                ok = false;
                break;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<ulonglong2*>(stage_row + ((u ^ (lane & 7)) << 4)) =
                    make_ulonglong2(sc2[2 * u], sc2[2 * u + 1]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                bulk_copy_to_cluster(peer_slice, smem_u32(sXs + widx * 4096), 4096u, peer_full);
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&xw_full[widx]), j & 1))) {
                ok = false;
                break;
            }
            // full scores: own + peer partial (IEEE addition commutes, so both CTAs
            // get the same bits)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(recv_row + ((u ^ (lane & 7)) << 4));
                sc2[2 * u] = add_f32x2(sc2[2 * u], x.x);
                sc2[2 * u + 1] = add_f32x2(sc2[2 * u + 1], x.y);
            }
            // X is consumed (its values are in registers): hand it back to the
            // peer.  A relaxed arrive: the peer only learns that the slice was
            // read, and a releasing one would wait for this warp's earlier
            // memory operations to complete first.
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote_relaxed(peer_free);

            // ---- scores in base 2, one packed FMA per token pair: score * (token
            // scale * softmax scale * log2 e) + (0, or -inf for a slot with no token;
            // its gathered row is zero, so its score is 0 and the FMA gives -inf)
            const int lb = j % kLatBufs;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&lat_full[lb]), (j / kLatBufs) & 1))) {
                ok = false;
                break;
            }
            const ulonglong2* mul4 = reinterpret_cast<const ulonglong2*>(sMult + lb * kNT + tcol);
            const ulonglong2* bia4 = reinterpret_cast<const ulonglong2*>(sBias + lb * kNT + tcol);
            float mh0 = -INFINITY, mh1 = -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const ulonglong2 mu = mul4[u], bi = bia4[u];
                sc2[2 * u] = fma_f32x2(sc2[2 * u], mu.x, bi.x);
                sc2[2 * u + 1] = fma_f32x2(sc2[2 * u + 1], mu.y, bi.y);
                const float2 a = unpack_f32x2(sc2[2 * u]), b = unpack_f32x2(sc2[2 * u + 1]);
                mh0 = fmaxf(mh0, fmaxf(a.x, b.x));
                mh1 = fmaxf(mh1, fmaxf(a.y, b.y));
            }
            const float m_half = fmaxf(mh0, mh1);
            // block max of the head over both halves
            sMax[half * 128 + h] = m_half;
            if (!pair_sync()) {
                ok = false;
                break;
            }
            const float m_blk = fmaxf(sMax[h], sMax[128 + h]);
            const float m_new = fmaxf(m_run, m_blk);
            // lazily refreshed running max: a head moves its max only when it grew
            // by more than 2^8 (both threads of the head decide alike); the O
            // rescale runs for the whole warp (factor 1 on lanes whose max stays)
            // because TMEM access is warp-collective, each thread of the pair
            // scaling its half of the columns
            float f = 1.f;
            if (m_new > m_run + kRescaleLog2) {
                if (m_run != -INFINITY) {
                    f = exp2f(m_run - m_new);
                    l_run *= f;
                }
                m_run = m_new;
            }
            if (__any_sync(0xffffffffu, f != 1.f)) {
                // j > 0 here: O holds blocks < j; PV(j - 1) has to complete before O
                // is rescaled
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(p_empty), (j - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t o[16];                       // 16 columns at a time: the scores stay in registers
                    const uint32_t col = 256 + half * 128 + c * 16;
                    tmem_ld_32x32b_x16(tmem_base + lane_base + col, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                    tmem_st_32x32b_x16(tmem_base + lane_base + col, o);
                }
                tmem_st_wait();
            }
            // P (f16, token scale folded in for V) -> TMEM lane h, over this block's
            // S columns: token pair (t, t + 1) of this thread's half in column
            // sb * 64 + half * 16 + t / 2 (both threads of the pair have read
            // their scores: the pair sync above ordered their loads)
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            const uint64_t negm = pack_f32x2(-m_use, -m_use);
            const ulonglong2* scl4 = reinterpret_cast<const ulonglong2*>(sScale + lb * kNT + tcol);
            uint64_t l2 = pack_f32x2(0.f, 0.f);
            uint32_t pk[16];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const ulonglong2 sv = scl4[u];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float2 d = unpack_f32x2(add_f32x2(sc2[2 * u + e], negm));
                    const uint64_t pp = pack_f32x2(ex2_approx(d.x), ex2_approx(d.y));   // -inf -> 0
                    l2 = add_f32x2(l2, pp);
                    const float2 pv = unpack_f32x2(mul_f32x2(pp, e == 0 ? sv.x : sv.y));
                    const __half2 b = __floats2half2_rn(pv.x, pv.y);
                    pk[2 * u + e] = *reinterpret_cast<const uint32_t*>(&b);
                }
            }
            const float2 lp = unpack_f32x2(l2);
            l_run += lp.x + lp.y;
            tmem_st_32x32b_x16(tmem_base + lane_base + sb * kNT + half * 16, pk);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&p_full[sb]));
        }
        if (!ok)
            *s_abort = 1;
        // ---- epilogue: O / l -> bf16 out[row][h][crank*256 + half*128 + v], lse (natural log)
        sSum[half * 128 + h] = l_run;
        const bool paired = ok && pair_sync();
        const float l_tot = sSum[h] + sSum[128 + h];
        const bool have = __all_sync(0xffffffffu, nblk > 0 && paired && mbar_wait(smem_u32(o_done), 0) && !*s_abort);
        tc_fence_after_sync();
        const float inv = (have && l_tot > 0.f) ? 1.f / l_tot : 0.f;
        __nv_bfloat16* orow = p.out + (static_cast<int64_t>(row) * p.num_heads + h) * 512 + crank * 256 + half * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            if (have) {                                   // warp-uniform: all lanes load
                tmem_ld_32x32b_x32(tmem_base + lane_base + 256 + half * 128 + c * 32, o);
                tmem_ld_wait();
            }
            if (h < p.num_heads) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint32_t pk[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const float a = have ? __uint_as_float(o[i + 2 * q2]) * inv : 0.f;
                        const float b = have ? __uint_as_float(o[i + 2 * q2 + 1]) * inv : 0.f;
                        const __nv_bfloat162 bb = __floats2bfloat162_rn(a, b);
                        pk[q2] = *reinterpret_cast<const uint32_t*>(&bb);
                    }
                    *reinterpret_cast<uint4*>(orow + c * 32 + i) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        }
        if (crank == 0 && half == 0 && h < p.num_heads)
            p.lse[static_cast<int64_t>(row) * p.num_heads + h] =
                (have && l_tot > 0.f) ? (m_run + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // every role is done: a wait that gave up anywhere in the CTA is visible now
    if (threadIdx.x == 0 && *s_abort && p.status)
        atomicOr(p.status, DSA_DEV_TIMEOUT);
    if (warp == kMmaWarp)
        tmem_dealloc(tmem_base, kTmemCols);
    cluster_sync();              // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

bool sparse_mla_tc_supported(const MlaArgs& a)
{
    return a.kv->fmt == DSA_KV_FP8_E4M3 && a.num_heads <= 128 && (a.d_qk == 576 || a.d_qk == 512) &&
           a.d_v == 512 && a.kv->sc_token_stride >= 4 && (!a.swa || a.swa->fmt == DSA_KV_FP8_E4M3);
}

dsa_status launch_sparse_mla_tc(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const dsa_paged_cache* kv = a.kv;
    constexpr MlaSmem mp = mla_smem();
    const int smem_bytes = static_cast<int>(mp.total) + 1024;
    if (smem_bytes > dev.max_smem_optin)
        return DSA_ERR_UNSUPPORTED;
    MlaParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.num_heads = a.num_heads;
    p.d_qk = a.d_qk;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.vals = static_cast<const uint8_t*>(kv->values);
    p.vps = kv->val_page_stride;
    p.vts = kv->val_token_stride;
    p.scs = static_cast<const uint8_t*>(kv->scales);
    p.sps = kv->sc_page_stride;
    p.sts = kv->sc_token_stride;
    p.bt = kv->block_table;
    p.bt_stride = kv->bt_row_stride;
    p.max_pages = kv->max_pages_per_seq;
    p.page_kv = kv->page_kv;
    p.num_pages = kv->num_pages;
    p.seq_of_row = a.seq_of_row;
    p.next_n = a.next_n;
    p.idx = a.idx;
    p.idx_stride = a.idx_row_stride;
    p.k = a.k;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.status = a.status;
    p.topk_lens = a.topk_lens;
    const dsa_paged_cache* w = a.swa;
    p.wvals = w ? static_cast<const uint8_t*>(w->values) : nullptr;
    p.wvps = w ? w->val_page_stride : 0;
    p.wvts = w ? w->val_token_stride : 0;
    p.wscs = w ? static_cast<const uint8_t*>(w->scales) : nullptr;
    p.wsps = w ? w->sc_page_stride : 0;
    p.wsts = w ? w->sc_token_stride : 0;
    p.wbt = w ? w->block_table : nullptr;
    p.wbt_stride = w ? w->bt_row_stride : 0;
    p.wmax_pages = w ? w->max_pages_per_seq : 0;
    p.wpage_kv = w ? w->page_kv : 1;
    p.wnum_pages = w ? w->num_pages : 0;
    p.window = w ? a.window : 0;
    p.seq_lens = a.seq_lens;
    p.cum_q = a.cum_q;
    p.batch = a.batch;
    const bool dual = a.topk_lens || a.swa || a.cum_q;
    auto kern = dual ? sparse_mla_tc_kernel<true> : sparse_mla_tc_kernel<false>;
    // q as [rows * num_heads][d_qk] bf16, boxes of 64 dims x 128 heads, 128B-swizzled
    CUtensorMap tm_q;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(a.d_qk), static_cast<uint64_t>(a.rows) * a.num_heads};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.d_qk) * 2};
        const uint32_t box[2] = {64, 128};
        const dsa_status st = encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dims, strides, box,
                                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != DSA_OK)
            return st;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e);
    // programmatic dependent launch: the launch overlaps the end of the
    // previous kernel, which the kernel waits for at entry
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, a.rows, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tm_q, p);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return check_launch();
}

}  // namespace dsa
