// topk.cu -- per-row top-k of the indexer logits by radix selection.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709): the indexer
// returns the top-k token positions per query row (indexer_score_topk), and
// the work is bounded by each row's ACTUAL visible length, not by the
// max-model-length width of the logits buffer.
//
// One CTA per row.  Logits are mapped to order-preserving uint32 keys; the k-th
// largest key is found with three histogram passes (11 + 11 + 10 bits) over the
// row, each pass only counting keys that match the digits already fixed; then
// one ordered pass writes every position with a larger key plus the first
// needed positions with an equal key (lowest positions win ties), ascending.
// The row is cached in shared memory when it fits (rows <= kSmemRowCap keys),
// otherwise every pass streams it from global memory (L2 after the first).
// Histogram updates are aggregated per warp (match.any) so that skewed digit
// distributions do not serialise on one shared-memory address.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"

namespace dsa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;
constexpr int kSmemRowCap = 40 * 1024;  // keys cached in shared memory (160 KB)

__device__ __forceinline__ uint32_t load_key(const float* row, int s)
{
    return float_key(__float_as_uint(__ldg(row + s)));
}

// Block-wide inclusive scan of one int per thread; returns inclusive value and
// the block total.  Uses ws[32] shared scratch.
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

template <bool kCached>
__global__ void __launch_bounds__(kTopkThreads, 1)
topk_kernel(const float* __restrict__ logits, int64_t stride, int width,
            const int32_t* __restrict__ context_lens, int next_n, int row_begin, int k,
            int32_t* __restrict__ idx, int64_t idx_stride, int32_t* __restrict__ count,
            int32_t* __restrict__ status)
{
    extern __shared__ uint32_t s_keys[];                 // [width] when kCached
    __shared__ int s_hist[kBins];
    __shared__ int s_ws[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;

    const int r = row_begin + blockIdx.x;
    const int b = r / next_n, i = r % next_n;
    int vis = visible_len(max(0, context_lens[b]), next_n, i);
    if (vis > width) {
        if (threadIdx.x == 0 && status)
            atomicOr(status, DSA_DEV_WIDTH);
        vis = width;
    }
    const float* row = logits + static_cast<int64_t>(blockIdx.x) * stride;
    int32_t* out = idx + static_cast<int64_t>(blockIdx.x) * idx_stride;
    const int take = vis < k ? vis : k;
    if (threadIdx.x == 0 && count)
        count[blockIdx.x] = take;

    if (vis <= k) {
        for (int s = threadIdx.x; s < k; s += kTopkThreads)
            out[s] = s < vis ? s : -1;
        return;
    }

    if (kCached) {
        // vectorised fill when the row start is 16-byte aligned
        const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
        int s0 = 0;
        if (vec) {
            const int nv = vis >> 2;
            const float4* row4 = reinterpret_cast<const float4*>(row);
            for (int v = threadIdx.x; v < nv; v += kTopkThreads) {
                const float4 x = __ldg(row4 + v);
                s_keys[4 * v + 0] = float_key(__float_as_uint(x.x));
                s_keys[4 * v + 1] = float_key(__float_as_uint(x.y));
                s_keys[4 * v + 2] = float_key(__float_as_uint(x.z));
                s_keys[4 * v + 3] = float_key(__float_as_uint(x.w));
            }
            s0 = nv << 2;
        }
        for (int s = s0 + threadIdx.x; s < vis; s += kTopkThreads)
            s_keys[s] = load_key(row, s);
    }

    auto key_at = [&](int s) -> uint32_t { return kCached ? s_keys[s] : load_key(row, s); };

    if (threadIdx.x == 0) {
        s_prefix = 0;
        s_need = k;
    }
    const int lane = threadIdx.x & 31;
    const int vis_warp = (vis + 31) & ~31;            // warp-uniform trip count
    // digits: bits [21,32), [10,21), [0,10)
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        for (int j = threadIdx.x; j < kBins; j += kTopkThreads)
            s_hist[j] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        const int sh = shifts[pass];
        const int hi = sh + widths[pass];             // bits above the digit are fixed
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int s = threadIdx.x; s < vis_warp; s += kTopkThreads) {
            int bin = -1;
            if (s < vis) {
                const uint32_t key = key_at(s);
                const bool match = (hi >= 32) ? true : ((key >> hi) == prefix);
                if (match)
                    bin = static_cast<int>((key >> sh) & dmask);
            }
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(peers) - 1)
                atomicAdd(&s_hist[bin], __popc(peers));
        }
        __syncthreads();
        // find the bin holding the need-th largest key: suffix counts from the top
        const int need = s_need;
        const int per = kBins / kTopkThreads;          // 2 bins per thread, top bins first
        int local = 0;
        for (int q = 0; q < per; ++q)
            local += s_hist[kBins - 1 - (threadIdx.x * per + q)];
        int total;
        const int incl = block_incl_scan(local, s_ws, &total);
        int before = incl - local;                     // keys in bins above this thread's
        if (before < need && need <= incl) {
            for (int q = 0; q < per; ++q) {
                const int bin = kBins - 1 - (threadIdx.x * per + q);
                const int c = s_hist[bin];
                if (before + c >= need) {
                    s_prefix = (prefix << widths[pass]) | static_cast<uint32_t>(bin);
                    s_need = need - before;
                    break;
                }
                before += c;
            }
        }
        __syncthreads();
    }
    const uint32_t thr = s_prefix;
    const int need_eq = s_need;                        // equal keys still to take

    // ordered output: keys > thr, plus the first need_eq keys == thr by position
    int written = 0, eq_seen = 0;
    for (int base = 0; base < vis; base += kTopkThreads) {
        const int s = base + threadIdx.x;
        uint32_t key = 0;
        if (s < vis)
            key = key_at(s);
        const int is_eq = (s < vis && key == thr) ? 1 : 0;
        int eq_tot;
        const int eq_incl = block_incl_scan(is_eq, s_ws, &eq_tot);
        const int sel = (s < vis) && (key > thr || (is_eq && eq_seen + eq_incl - 1 < need_eq)) ? 1 : 0;
        int sel_tot;
        const int sel_incl = block_incl_scan(sel, s_ws, &sel_tot);
        if (sel)
            out[written + sel_incl - 1] = s;
        written += sel_tot;
        eq_seen += eq_tot;
    }
    for (int s = written + threadIdx.x; s < k; s += kTopkThreads)
        out[s] = -1;
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
