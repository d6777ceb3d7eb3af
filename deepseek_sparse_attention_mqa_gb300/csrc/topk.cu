// topk.cu -- per-row top-k of the indexer logits.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709): the indexer
// returns the top-k token positions per query row (indexer_score_topk), and
// the work is bounded by each row's ACTUAL visible length, not by the
// max-model-length width of the logits buffer.
//
// One CTA per row.  Logits are mapped to order-preserving uint32 keys.  The
// row's key range [kmin, kmax] is split into 2048 bins by a right shift, which
// bins in bit-pattern space: uniform in log scale, so outliers and wide value
// ranges cost nothing.  One histogram pass finds the bin holding the k-th
// largest key (refined with narrower bins while that bin is crowded), then one
// output pass writes every position above that bin and collects the bin's few
// elements as candidates, which are resolved exactly by the 64-bit order
// (key, then lower position first) -- the same order as a full sort with ties
// broken by position.  The row is kept in shared memory when it fits.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"

namespace dsa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;
constexpr int kBinBits = 11;
constexpr int kCandCap = 4096;          // threshold-bin candidates kept in shared memory
constexpr int kRankCap = 1024;          // candidates resolved by direct ranking
constexpr int kSmemRowCap = 40 * 1024;  // keys cached in shared memory (160 KB)

__device__ __forceinline__ uint64_t order64(uint32_t key, int pos)
{
    // larger key first, then lower position first
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(pos));
}

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
        int t = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    *total = ws[31];
    return x + (warp > 0 ? ws[warp - 1] : 0);
}

// Warp-aggregated append: returns the slot of this lane's element (or -1).
__device__ __forceinline__ int warp_append(bool take, int* counter)
{
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (!m)
        return -1;
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == __ffs(m) - 1)
        base = atomicAdd(counter, __popc(m));
    base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
    return take ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

template <bool kCached>
__global__ void __launch_bounds__(kTopkThreads, 1)
topk_kernel(const float* __restrict__ logits, int64_t stride, int width,
            const int32_t* __restrict__ context_lens, int next_n, int row_begin, int k,
            int32_t* __restrict__ idx, int64_t idx_stride, int32_t* __restrict__ count,
            int32_t* __restrict__ status)
{
    extern __shared__ uint32_t s_keys[];                 // [width] when kCached
    __shared__ int s_hist[kBins];
    __shared__ uint32_t s_ck[kCandCap];
    __shared__ int s_cp[kCandCap];
    __shared__ int s_ws[32];
    __shared__ int s_bin, s_above_bin;
    __shared__ int s_nout, s_ncand;
    __shared__ unsigned s_kmin, s_kmax;

    const int tid = threadIdx.x, lane = tid & 31;
    const int r = row_begin + blockIdx.x;
    const int b = r / next_n, i = r % next_n;
    int vis = visible_len(max(0, context_lens[b]), next_n, i);
    if (vis > width) {
        if (tid == 0 && status)
            atomicOr(status, DSA_DEV_WIDTH);
        vis = width;
    }
    const float* row = logits + static_cast<int64_t>(blockIdx.x) * stride;
    int32_t* out = idx + static_cast<int64_t>(blockIdx.x) * idx_stride;
    const int take = vis < k ? vis : k;
    if (tid == 0 && count)
        count[blockIdx.x] = take;
    if (vis <= k) {
        for (int s = tid; s < k; s += kTopkThreads)
            out[s] = s < vis ? s : -1;
        return;
    }

    // ---- keys (cached) and key range
    if (tid == 0) {
        s_kmin = 0xFFFFFFFFu;
        s_kmax = 0u;
        s_nout = 0;
        s_ncand = 0;
    }
    __syncthreads();
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    {
        const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
        int s0 = 0;
        if (vec) {
            const int nv = vis >> 2;
            const float4* row4 = reinterpret_cast<const float4*>(row);
            for (int v = tid; v < nv; v += kTopkThreads) {
                const float4 x = __ldg(row4 + v);
                const uint32_t a = float_key(__float_as_uint(x.x)), bb = float_key(__float_as_uint(x.y));
                const uint32_t c = float_key(__float_as_uint(x.z)), d = float_key(__float_as_uint(x.w));
                if (kCached) {
                    s_keys[4 * v + 0] = a;
                    s_keys[4 * v + 1] = bb;
                    s_keys[4 * v + 2] = c;
                    s_keys[4 * v + 3] = d;
                }
                kmin = min(kmin, min(min(a, bb), min(c, d)));
                kmax = max(kmax, max(max(a, bb), max(c, d)));
            }
            s0 = nv << 2;
        }
        for (int s = s0 + tid; s < vis; s += kTopkThreads) {
            const uint32_t a = float_key(__float_as_uint(__ldg(row + s)));
            if (kCached)
                s_keys[s] = a;
            kmin = min(kmin, a);
            kmax = max(kmax, a);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) {
        atomicMin(&s_kmin, kmin);
        atomicMax(&s_kmax, kmax);
    }
    __syncthreads();
    auto key_at = [&](int s) -> uint32_t {
        return kCached ? s_keys[s] : float_key(__float_as_uint(__ldg(row + s)));
    };

    // ---- histogram passes: find the bin of the k-th largest key
    uint32_t lo = s_kmin, hi = s_kmax;
    int need = k;                 // still to take from keys in [lo, hi]
    int shift = 0;
    while (true) {
        const uint64_t span = static_cast<uint64_t>(hi) - lo + 1;
        shift = max(0, log2_ceil_u64(span) - kBinBits);
        for (int j = tid; j < kBins; j += kTopkThreads)
            s_hist[j] = 0;
        __syncthreads();
        for (int s = tid; s < vis; s += kTopkThreads) {
            const uint32_t key = key_at(s);
            if (key >= lo && key <= hi)
                atomicAdd(&s_hist[(key - lo) >> shift], 1);
        }
        __syncthreads();
        // suffix counts from the top bin down: thread t owns bins 2047-2t, 2046-2t
        const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
        const int c0 = s_hist[b0], c1 = s_hist[b1];
        int total;
        const int incl = block_incl_scan(c0 + c1, s_ws, &total);
        const int before = incl - c0 - c1;
        if (before < need && need <= incl) {
            if (before + c0 >= need) {
                s_bin = b0;
                s_above_bin = before;
            } else {
                s_bin = b1;
                s_above_bin = before + c0;
            }
        }
        __syncthreads();
        const int bin = s_bin;
        need -= s_above_bin;
        const uint32_t blo = lo + (static_cast<uint32_t>(bin) << shift);
        const uint32_t bhi = static_cast<uint32_t>(
            min(static_cast<uint64_t>(hi), static_cast<uint64_t>(blo) + ((uint64_t(1) << shift) - 1)));
        const int in_bin = s_hist[bin];
        __syncthreads();
        if (in_bin <= kCandCap || shift == 0) {
            lo = blo;
            hi = bhi;
            break;
        }
        lo = blo;                 // crowded bin: refine inside it
        hi = bhi;
    }
    // keys > hi are taken outright (k - need of them); keys in [lo, hi] are candidates
    const int n_direct = k - need;

    // ---- output pass
    int cand_total;
    {
        for (int base = 0; base < vis; base += kTopkThreads) {
            const int s = base + tid;
            uint32_t key = 0;
            if (s < vis)
                key = key_at(s);
            const bool above = s < vis && key > hi;
            const bool cand = s < vis && key >= lo && key <= hi;
            const int slot = warp_append(above, &s_nout);
            if (slot >= 0)
                out[slot] = s;
            const int cs = warp_append(cand, &s_ncand);
            if (cs >= 0 && cs < kCandCap) {
                s_ck[cs] = key;
                s_cp[cs] = s;
            }
        }
        __syncthreads();
        cand_total = s_ncand;
    }

    // ---- resolve the candidates: the `need` best by (key desc, position asc)
    if (cand_total <= kCandCap) {
        if (cand_total <= kRankCap) {
            if (tid < cand_total) {
                const uint64_t me = order64(s_ck[tid], s_cp[tid]);
                int rank = 0;
                for (int j = 0; j < cand_total; ++j)
                    rank += order64(s_ck[j], s_cp[j]) > me ? 1 : 0;
                if (rank < need)
                    out[n_direct + rank] = s_cp[tid];
            }
        } else {
            // radix selection on the 64-bit order, 8 bits at a time (high to low)
            uint64_t prefix = 0;
            int rem = need;
            for (int pass = 7; pass >= 0; --pass) {
                const int sh = 8 * pass;
                for (int j = tid; j < 256; j += kTopkThreads)
                    s_hist[j] = 0;
                __syncthreads();
                for (int j = tid; j < cand_total; j += kTopkThreads) {
                    const uint64_t o = order64(s_ck[j], s_cp[j]);
                    const bool match = (pass == 7) || ((o >> (sh + 8)) == (prefix >> (sh + 8)));
                    if (match)
                        atomicAdd(&s_hist[(o >> sh) & 255], 1);
                }
                __syncthreads();
                if (tid == 0) {
                    int acc = 0;
                    for (int d = 255; d >= 0; --d) {
                        if (acc + s_hist[d] >= rem) {
                            s_bin = d;
                            s_above_bin = acc;
                            break;
                        }
                        acc += s_hist[d];
                    }
                }
                __syncthreads();
                prefix |= static_cast<uint64_t>(s_bin) << sh;
                rem -= s_above_bin;
                __syncthreads();
            }
            // order values are unique: take every candidate >= prefix
            if (tid == 0)
                s_nout = n_direct;
            __syncthreads();
            for (int base = 0; base < cand_total; base += kTopkThreads) {
                const int j = base + tid;
                const bool t = j < cand_total && order64(s_ck[j], s_cp[j]) >= prefix;
                const int slot = warp_append(t, &s_nout);
                if (slot >= 0)
                    out[slot] = s_cp[j];
            }
        }
    } else {
        // only when every candidate has one key value (shift == 0): take the
        // `need` lowest positions holding it, in position order
        const uint32_t key_eq = lo;
        int seen = 0;
        for (int base = 0; base < vis && seen < need; base += kTopkThreads) {
            const int s = base + tid;
            const int is_eq = (s < vis && key_at(s) == key_eq) ? 1 : 0;
            int tot;
            const int incl = block_incl_scan(is_eq, s_ws, &tot);
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
    (void)dev;
    const int rows = a.row_end - a.row_begin;
    if (rows <= 0)
        return DSA_OK;
    const float* lg = a.logits;
    if (a.logits_width <= kSmemRowCap) {
        const int smem = a.logits_width * 4;
        cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        topk_kernel<true><<<rows, kTopkThreads, smem, stream>>>(
            lg, a.logits_row_stride, a.logits_width, a.context_lens, a.next_n, a.row_begin, a.k, a.idx,
            a.idx_row_stride, a.count, a.status);
    } else {
        topk_kernel<false><<<rows, kTopkThreads, 0, stream>>>(
            lg, a.logits_row_stride, a.logits_width, a.context_lens, a.next_n, a.row_begin, a.k, a.idx,
            a.idx_row_stride, a.count, a.status);
    }
    return check_launch();
}

}  // namespace dsa
