// topk.cu -- per-row top-k of the indexer logits.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709): the indexer
// returns the top-k token positions per query row (indexer_score_topk), and
// the work is bounded by each row's ACTUAL visible length, not by the
// max-model-length width of the logits buffer.
//
// A cluster of C CTAs per row (C = 1..8, chosen so that all SMs have work even
// for a 64-row decode batch); CTA c owns a contiguous slice of the row, keeps it
// in shared memory as order-preserving uint32 keys, and the cluster cooperates
// through distributed shared memory (CTA 0 collects the output counters and
// the candidates):
//  1. the slice's keys into shared memory; the barrier that publishes the
//     zeroed counters to the cluster is split around this load (arrive before,
//     wait after the first local histogram), so its latency is hidden;
//  2. 2048 bins by a right shift, the first round over the whole key space (the
//     key's top 11 bits) -- bins uniform in bit-pattern space, i.e. log scale,
//     so outliers and wide ranges cost nothing; one histogram round finds the
//     bin of the k-th largest key, refined inside that bin while it is
//     crowded.  Each CTA adds its counts into every CTA's copy of the row
//     histogram, so after one cluster barrier every CTA scans the same counts
//     and takes the same decision, with no broadcast and no second barrier;
//  3. every position above that bin is written out directly (cluster-wide
//     counter); the bin's few elements are appended to CTA 0 as candidates;
//  4. CTA 0 resolves the candidates exactly by the 64-bit order (key, then lower
//     position), the same order as a full sort with ties broken by position:
//     by ranking each candidate against the others when there are at most 256,
//     else with a parallel radix selection (11-bit digits, block-wide scans).
// A launch with one CTA per row (C = 1, prefill chunks) runs its own
// instantiation, with block barriers and local shared memory in place of the
// cluster's barriers and distributed shared memory.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kBins = 2048;
constexpr int kBinBits = 11;
constexpr int kCandCap = 4096;      // threshold-bin candidates collected in CTA 0
constexpr int kRankSelectMax = 256; // up to this many candidates are selected by direct ranking
constexpr int kSliceCap = 16384;    // keys per CTA kept in shared memory (64 KB)
constexpr int kMaxCluster = 8;

__device__ __forceinline__ int log2_ceil_u64(uint64_t v)
{
    return v <= 1 ? 0 : 64 - __clzll(v - 1);
}

// Block-wide inclusive scan of one int per thread (uses ws[32]).
__device__ __forceinline__ int block_incl_scan(int v, int* ws, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    __syncthreads();
    if (lane == 31)
        ws[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kThreads / 32 ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    *total = ws[kThreads / 32 - 1];
    return x + (warp > 0 ? ws[warp - 1] : 0);
}

struct TopkShared {
    int hist[kBins];              // the row's histogram: every CTA adds its counts into every CTA's copy
    uint32_t ck[kCandCap];
    int cp[kCandCap];             // also this CTA's own histogram during the rounds
    int ws[32];
    int bin, above, in_bin;       // histogram decision (taken by every CTA alike)
    int nout, ncand;
    int res_above, res_cand;      // this CTA's reserved output / candidate ranges
};

// two CTAs per SM: a decode batch's clusters (e.g. 64 rows x 4 CTAs) fit in one wave
template <bool kCached, bool kSolo>
__global__ void __launch_bounds__(kThreads, 2)
topk_kernel(const float* __restrict__ logits, int64_t stride, int width,
            const int32_t* __restrict__ context_lens, int next_n, int ratio, int row_begin, int k,
            int32_t* __restrict__ idx, int64_t idx_stride, int32_t* __restrict__ count,
            int32_t* __restrict__ status)
{
    extern __shared__ uint32_t s_keys[];                 // [slice] when kCached
    __shared__ TopkShared sh;

    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t crank = cluster_ctarank();
    const int C = static_cast<int>(gridDim.x);           // cluster spans gridDim.x
    // kSolo (launched with C = 1): a row handled by one CTA, with block
    // barriers and local shared memory instead of the cluster's
    constexpr bool solo = kSolo;

    // Everything another CTA touches remotely (every CTA's first-round row
    // histogram, CTA 0's output and candidate counters) is initialised before
    // the first cluster barrier: arrived at here, waited on after the first
    // local histogram.  This touches shared memory only, so it runs before the
    // wait below, while the previous kernel finishes.
    int* own = sh.cp;                                     // this CTA's histogram (candidates come later)
    if (tid == 0) {
        sh.nout = 0;
        sh.ncand = 0;
    }
    for (int j = tid; j < kBins; j += kThreads) {
        sh.hist[j] = 0;
        own[j] = 0;
    }
    __syncthreads();
    if (!solo)
        cluster_arrive();

    // launched as a programmatic dependent of the previous kernel of the stream:
    // nothing it may have written is read before this wait (the launch latency
    // and the set-up above are what overlap); the MLA that follows may then
    // start its blocks
    pdl_wait();
    pdl_launch_dependents();
    const int rloc = blockIdx.y;
    const int r = row_begin + rloc;
    const int b = r / next_n, i = r % next_n;
    int vis = visible_entries(max(0, context_lens[b]), next_n, i, ratio);
    if (vis > width) {
        if (tid == 0 && crank == 0 && status)
            atomicOr(status, DSA_DEV_WIDTH);
        vis = width;
    }
    const float* row = logits + static_cast<int64_t>(rloc) * stride;
    int32_t* out = idx + static_cast<int64_t>(rloc) * idx_stride;
    if (vis <= k) {                                       // uniform over the cluster
        if (crank == 0) {
            if (tid == 0 && count)
                count[rloc] = vis;
            for (int s = tid; s < k; s += kThreads)
                out[s] = s < vis ? s : -1;
        }
        if (!solo)
            cluster_wait();                               // the arrive above is matched before leaving
        return;
    }

    // this CTA's slice [s_lo, s_hi) of the visible row (slice starts 16-byte aligned)
    const int slice = (((vis + C - 1) / C) + 3) & ~3;
    const int s_lo = min(vis, static_cast<int>(crank) * slice);
    const int s_hi = min(vis, s_lo + slice);
    const int n = s_hi - s_lo;

    // CTA 0's copies of the shared reduction state (cluster addresses)
    const uint32_t c0_nout = mapa_shared(smem_u32(&sh.nout), 0);
    const uint32_t c0_ncand = mapa_shared(smem_u32(&sh.ncand), 0);
    const uint32_t c0_ck = mapa_shared(smem_u32(&sh.ck[0]), 0);
    const uint32_t c0_cp = mapa_shared(smem_u32(&sh.cp[0]), 0);

    // ---- 1. keys of the slice, counted into the first round's local histogram
    // as they are loaded (that round's bins are the key's top 11 bits)
    constexpr int kFirstShift = 32 - kBinBits;
    {
        const float* src = row + s_lo;
        const bool vec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0);
        int s0 = 0;
        if (vec) {
            const int nv = n >> 2;
            const float4* src4 = reinterpret_cast<const float4*>(src);
            for (int v = tid; v < nv; v += kThreads) {
                const float4 x = __ldg(src4 + v);
                const uint32_t a = float_key(__float_as_uint(x.x)), bb = float_key(__float_as_uint(x.y));
                const uint32_t c = float_key(__float_as_uint(x.z)), d = float_key(__float_as_uint(x.w));
                if (kCached) {
                    s_keys[4 * v + 0] = a;
                    s_keys[4 * v + 1] = bb;
                    s_keys[4 * v + 2] = c;
                    s_keys[4 * v + 3] = d;
                }
                atomicAdd(&own[a >> kFirstShift], 1);
                atomicAdd(&own[bb >> kFirstShift], 1);
                atomicAdd(&own[c >> kFirstShift], 1);
                atomicAdd(&own[d >> kFirstShift], 1);
            }
            s0 = nv << 2;
        }
        for (int s = s0 + tid; s < n; s += kThreads) {
            const uint32_t a = float_key(__float_as_uint(__ldg(src + s)));
            if (kCached)
                s_keys[s] = a;
            atomicAdd(&own[a >> kFirstShift], 1);
        }
    }
    __syncthreads();                                      // keys and first-round counts are in place
    auto key_at = [&](int j) -> uint32_t {               // j: index within the slice
        return kCached ? s_keys[j] : float_key(__float_as_uint(__ldg(row + s_lo + j)));
    };
    uint32_t lo = 0u, hi = 0xFFFFFFFFu;

    // ---- 2. histogram rounds: the bin of the k-th largest key.  Each CTA adds
    // its counts into every CTA's row histogram, so after one cluster barrier
    // every CTA scans the same histogram and takes the same decision itself.
    int need = k;                 // still to take from keys in [lo, hi]
    for (int round = 0;; ++round) {
        const uint64_t span = static_cast<uint64_t>(hi) - lo + 1;
        const int shift = max(0, log2_ceil_u64(span) - kBinBits);
        if (round > 0) {
            // (the first round's histograms were zeroed before the first barrier;
            // each CTA has read its row histogram for the last decision)
            for (int j = tid; j < kBins; j += kThreads) {
                sh.hist[j] = 0;
                own[j] = 0;
            }
            if (solo)
                __syncthreads();
            else
                cluster_sync();                           // every row histogram zeroed
            for (int j = tid; j < n; j += kThreads) {
                const uint32_t key = key_at(j);
                if (key >= lo && key <= hi)
                    atomicAdd(&own[(key - lo) >> shift], 1);
            }
            __syncthreads();
        } else {
            // (this CTA's first-round counts were taken as its keys were loaded)
            if (!solo)
                cluster_wait();                           // every CTA's counters are zeroed
        }
        for (int j = tid; j < kBins; j += kThreads) {
            const int v = own[j];
            if (v && solo) {
                sh.hist[j] = v;
            } else if (v) {
                const uint32_t a = smem_u32(&sh.hist[j]);
                for (int cr = 0; cr < C; ++cr)
                    red_add_cluster(mapa_shared(a, static_cast<uint32_t>(cr)), static_cast<uint32_t>(v));
            }
        }
        if (solo)
            __syncthreads();
        else
            cluster_sync();                               // every CTA holds the row histogram
        {
            // suffix counts from the top bin down: thread t owns bins 2047-4t .. 2044-4t
            int c[4], loc = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                c[q] = sh.hist[kBins - 1 - 4 * tid - q];
                loc += c[q];
            }
            int total;
            const int incl = block_incl_scan(loc, sh.ws, &total);
            int before = incl - loc;
            if (before < need && need <= incl) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (before + c[q] >= need) {
                        sh.bin = kBins - 1 - 4 * tid - q;
                        sh.above = before;
                        sh.in_bin = c[q];
                        break;
                    }
                    before += c[q];
                }
            }
        }
        __syncthreads();                                  // the decision
        const int bin = sh.bin;
        need -= sh.above;
        const int in_bin = sh.in_bin;
        const uint32_t blo = lo + (static_cast<uint32_t>(bin) << shift);
        const uint32_t bhi = static_cast<uint32_t>(
            min(static_cast<uint64_t>(hi), static_cast<uint64_t>(blo) + ((uint64_t(1) << shift) - 1)));
        lo = blo;
        hi = bhi;
        if (in_bin <= kCandCap || shift == 0)
            break;
    }
    const int n_direct = k - need;                        // keys > hi are taken outright

    // ---- 3. output pass: keys above the bin out, the bin's keys to CTA 0 as
    // candidates.  Each CTA counts first and reserves its ranges with one
    // cluster atomic per counter, then writes at thread-local offsets.
    int n_above = 0, n_cand = 0;
    for (int j = tid; j < n; j += kThreads) {
        const uint32_t key = key_at(j);
        n_above += key > hi ? 1 : 0;
        n_cand += (key >= lo && key <= hi) ? 1 : 0;
    }
    int tot_above, tot_cand, off_above, off_cand;
    if (n < 65536) {
        // both counts in one scan: above in bits 0-15, candidates in bits 16-31
        int tot;
        const int v = n_above | (n_cand << 16);
        const uint32_t ex = static_cast<uint32_t>(block_incl_scan(v, sh.ws, &tot) - v);
        off_above = static_cast<int>(ex & 0xFFFFu);
        off_cand = static_cast<int>(ex >> 16);
        tot_above = static_cast<int>(static_cast<uint32_t>(tot) & 0xFFFFu);
        tot_cand = static_cast<int>(static_cast<uint32_t>(tot) >> 16);
    } else {
        off_above = block_incl_scan(n_above, sh.ws, &tot_above) - n_above;
        off_cand = block_incl_scan(n_cand, sh.ws, &tot_cand) - n_cand;
    }
    if (tid == 0 && solo) {
        sh.res_above = 0;
        sh.res_cand = 0;
        sh.nout = tot_above;
        sh.ncand = tot_cand;
    } else if (tid == 0) {
        sh.res_above = tot_above ? static_cast<int>(atom_add_cluster(c0_nout, static_cast<uint32_t>(tot_above))) : 0;
        sh.res_cand = tot_cand ? static_cast<int>(atom_add_cluster(c0_ncand, static_cast<uint32_t>(tot_cand))) : 0;
    }
    __syncthreads();
    // The candidates go to CTA 0 first and the barrier that publishes them is
    // arrived at before the positions above the bin are written: its release
    // then waits only for the shared-memory stores, not for the global ones.
    {
        int oc = sh.res_cand + off_cand;
        for (int j = tid; j < n; j += kThreads) {
            const uint32_t key = key_at(j);
            if (key >= lo && key <= hi) {
                if (oc < kCandCap && solo) {
                    sh.ck[oc] = key;
                    sh.cp[oc] = s_lo + j;
                } else if (oc < kCandCap) {
                    st_cluster_u32(c0_ck + 4u * oc, key);
                    st_cluster_u32(c0_cp + 4u * oc, static_cast<uint32_t>(s_lo + j));
                }
                ++oc;
            }
        }
    }
    if (!solo)
        cluster_arrive();
    {
        int oa = sh.res_above + off_above;
        for (int j = tid; j < n; j += kThreads)
            if (key_at(j) > hi)
                out[oa++] = s_lo + j;
    }
    if (solo)
        __syncthreads();
    else
        cluster_wait();                                   // all candidates landed in CTA 0
    if (crank != 0)
        return;
    if (tid == 0 && count)
        count[rloc] = k;

    // ---- 4. CTA 0: the `need` best candidates by (key desc, position asc).
    // Radix selection on o = (key - lo) << 32 | ~position, 11 bits at a time
    // from the top, each digit found by a block-wide scan of the digit
    // histogram; it stops as soon as the chosen digit's bin holds exactly the
    // number still needed (then every candidate matching the prefix is in).
    const int cand_total = sh.ncand;
    auto cand_order = [&](int j) -> uint64_t {
        return (static_cast<uint64_t>(sh.ck[j] - lo) << 32) |
               static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(sh.cp[j]));
    };
    if (cand_total <= kRankSelectMax) {
        // Few candidates (the usual case: the threshold bin of a decode row holds
        // tens of keys): each thread ranks one candidate against all of them by
        // the same 64-bit order (unique: positions differ), and the `need` best
        // go straight to their slots -- no radix rounds, no block barriers.
        for (int t = tid; t < cand_total; t += kThreads) {
            const uint64_t ot = cand_order(t);
            int rank = 0;
            for (int j = 0; j < cand_total; ++j)
                rank += cand_order(j) > ot ? 1 : 0;
            if (rank < need)
                out[n_direct + rank] = sh.cp[t];
        }
    } else if (cand_total <= kCandCap) {
        const int key_bits = log2_ceil_u64(static_cast<uint64_t>(hi - lo) + 1);
        uint64_t prefix = 0;
        int rem = need;
        int top = 32 + key_bits;                          // bits [0, top) still undecided
        while (top > 0) {
            const int lo_bit = max(0, top - kBinBits);
            const uint64_t mask = (uint64_t(1) << (top - lo_bit)) - 1;
            for (int j = tid; j < kBins; j += kThreads)
                sh.hist[j] = 0;
            __syncthreads();
            for (int j = tid; j < cand_total; j += kThreads) {
                const uint64_t o = cand_order(j);
                if (top >= 64 || (o >> top) == (prefix >> top))
                    atomicAdd(&sh.hist[(o >> lo_bit) & mask], 1);
            }
            __syncthreads();
            // suffix counts from the top bin down: thread t owns bins 2047-4t .. 2044-4t
            int c[4], loc = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                c[q] = sh.hist[kBins - 1 - 4 * tid - q];
                loc += c[q];
            }
            int total;
            const int incl = block_incl_scan(loc, sh.ws, &total);
            int before = incl - loc;
            if (before < rem && rem <= incl) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (before + c[q] >= rem) {
                        sh.bin = kBins - 1 - 4 * tid - q;
                        sh.above = before;
                        sh.in_bin = c[q];
                        break;
                    }
                    before += c[q];
                }
            }
            __syncthreads();
            prefix |= static_cast<uint64_t>(sh.bin) << lo_bit;
            rem -= sh.above;
            const int in_bin = sh.in_bin;
            top = lo_bit;
            __syncthreads();
            if (in_bin == rem)
                break;                                    // the whole bin is taken
        }
        // selected: candidates whose bits [top, 64) are >= the prefix's
        if (tid == 0)
            sh.nout = n_direct;
        __syncthreads();
        for (int base = 0; base < cand_total; base += kThreads) {
            const int j = base + tid;
            const bool t = j < cand_total && (top >= 64 ? true : (cand_order(j) >> top) >= (prefix >> top));
            const unsigned m = __ballot_sync(0xffffffffu, t);
            int slot = 0;
            if (lane == __ffs(m) - 1)
                slot = atomicAdd(&sh.nout, __popc(m));
            slot = __shfl_sync(0xffffffffu, slot, m ? __ffs(m) - 1 : 0) + __popc(m & ((1u << lane) - 1u));
            if (t)
                out[slot] = sh.cp[j];
        }
    } else {
        // every candidate carries one key value (shift reached 0): take the
        // `need` lowest positions holding it, in position order
        const uint32_t key_eq = lo;
        int seen = 0;
        for (int base = 0; base < vis && seen < need; base += kThreads) {
            const int s = base + tid;
            const int is_eq = (s < vis && float_key(__float_as_uint(__ldg(row + s))) == key_eq) ? 1 : 0;
            int tot;
            const int incl = block_incl_scan(is_eq, sh.ws, &tot);
            const int rank = seen + incl - 1;
            if (is_eq && rank < need)
                out[n_direct + rank] = s;
            seen += tot;
        }
    }
}

}  // namespace

dsa_status launch_topk(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const int rows = a.row_end - a.row_begin;
    if (rows <= 0)
        return DSA_OK;
    // cluster size: enough CTAs to cover ~1.5x the SMs, at least enough that a
    // slice of the widest row fits in shared memory, at most 8
    int C = 1;
    while (C < kMaxCluster && (static_cast<int64_t>(a.logits_width) + C - 1) / C > kSliceCap)
        C <<= 1;
    while (C < kMaxCluster && static_cast<int64_t>(rows) * C * 2 < 3LL * dev.sm_count)
        C <<= 1;
    const int slice = static_cast<int>((((static_cast<int64_t>(a.logits_width) + C - 1) / C) + 3) & ~3LL);
    const bool cached = slice <= kSliceCap;
    const int smem = cached ? slice * 4 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, rows, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel's blocks may start while the
    // logits kernel finishes; they wait (griddepcontrol.wait) before reading it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    if (cached) {
        // one CTA per row (C = 1) gets its own instantiation without cluster operations
        auto kern = C == 1 ? topk_kernel<true, true> : topk_kernel<true, false>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        e = cudaLaunchKernelEx(&cfg, kern, a.logits, a.logits_row_stride, a.logits_width,
                               a.context_lens, a.next_n, a.ratio, a.row_begin, a.k, a.idx, a.idx_row_stride, a.count,
                               a.status);
    } else {
        // (a slice above the shared-memory cap happens only at the largest cluster)
        e = cudaLaunchKernelEx(&cfg, topk_kernel<false, false>, a.logits, a.logits_row_stride, a.logits_width,
                               a.context_lens, a.next_n, a.ratio, a.row_begin, a.k, a.idx, a.idx_row_stride, a.count,
                               a.status);
    }
    if (e != cudaSuccess)
        return cuda_fail(e);
    return check_launch();
}

}  // namespace dsa
