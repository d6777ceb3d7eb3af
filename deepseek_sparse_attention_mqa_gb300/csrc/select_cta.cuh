// select_cta.cuh -- top-k of one row by ONE thread block (all its threads).
//
// Used by the fused indexer score + top-k kernels: the block that finishes a
// row's last logits tile selects that row from the logits just written (in L2).
// Same result as a full sort of the row's visible logits by (logit descending,
// position ascending) -- -0 equals +0 -- by a radix/bin selection on the
// order-preserving uint32 images ("keys") of the logits:
//  1. one pass over the row (16-byte loads, eight in flight per thread) counts
//     the keys per 2048 bins of their top 11 bits and, when the row fits, keeps
//     the keys in shared memory;
//  2. the bin of the k-th largest key is found by a block-wide scan; while it
//     holds more keys than the candidate store, it is split again into 2048
//     bins by the next bits (from the cached keys, or another pass);
//  3. every thread counts its keys above the bin and in it, one block scan
//     gives each thread its offsets, and a second sweep writes the keys above
//     the bin to the output and the bin's keys to the candidate store (no
//     contended shared counter);
//  4. the candidates are resolved exactly by the 64-bit order (key, then lower
//     position): by ranking when there are at most 256, else by 8-bit radix
//     digits; a bin of one key value too large to store is taken in position
//     order.
// A cached row costs one pass over L2 and shared-memory passes after it; a row
// too long for the cache costs two passes (more only if its threshold bin
// overflows the candidate store).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dsa {

constexpr int kSelBins = 2048;
constexpr int kSelBinBits = 11;
constexpr int kSelRankMax = 256;
constexpr int kSelCandCached = 4096;    // candidate store beside a cached row
constexpr int kSelCandMax = 16384;      // candidate store of an uncached row
constexpr int kSelUnroll = 8;           // 16-byte loads in flight per thread

struct SelectSmem {
    int hist[kSelBins];
    int ws[33];
    int bin, above, in_bin;
    int nout, ncand;
    int pad[3];
};

__device__ __forceinline__ int sel_log2_ceil(uint64_t v)
{
    return v <= 1 ? 0 : 64 - __clzll(v - 1);
}

// Inclusive scan of one int per thread over the whole block (blockDim.x <= 1024).
__device__ __forceinline__ int sel_block_scan(int v, int* ws, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = (blockDim.x + 31) >> 5;
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
        int t = lane < nw ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    *total = ws[nw - 1];
    return x + (warp > 0 ? ws[warp - 1] : 0);
}

// The bin of hist[0 : nbins) holding the need-th largest element, counted
// from the top bin down: sets sh.bin, sh.above (elements in higher bins) and
// sh.in_bin.  nbins is 2048 or 256: threads t < 256 own nbins/256 consecutive
// bins each (their loads independent), one block scan orders the owners.  All
// threads call it; 1 <= need <= total count.
__device__ __forceinline__ void sel_find_bin(SelectSmem& sh, const int* hist, int nbins, int need)
{
    const int t = threadIdx.x;
    const int per = nbins >> 8;                    // 8 or 1
    int c[8];
    int loc = 0;
    if (t < 256) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            c[q] = q < per ? hist[nbins - 1 - per * t - q] : 0;
            loc += c[q];
        }
    }
    int total;
    const int incl = sel_block_scan(t < 256 ? loc : 0, sh.ws, &total);
    if (t < 256) {
        int before = incl - loc;
        if (before < need && need <= incl) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < per && before + c[q] >= need) {
                    sh.bin = nbins - 1 - per * t - q;
                    sh.above = before;
                    sh.in_bin = c[q];
                    break;
                }
                before += c[q];
            }
        }
    }
    __syncthreads();
}

// Calls f(j, key, valid) for every position j < n of the row, reading it from
// global memory (L2) with kSelUnroll 16-byte loads in flight per thread.  Every
// thread of the block makes the same sequence of calls (valid = false past the
// end), so f may use warp votes.  The row must be 16-byte aligned.
template <class F>
__device__ __forceinline__ void sel_stream_row(const float* __restrict__ row, int n, F&& f)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nv = (n + 3) >> 2;                              // float4s, the last one partial
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int base = 0; base < nv; base += nt * kSelUnroll) {
        float4 x[kSelUnroll];
#pragma unroll
        for (int u = 0; u < kSelUnroll; ++u) {
            const int v = base + u * nt + tid;
            x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * v + 3 < n) {
                x[u] = __ldcg(r4 + v);
            } else if (v < nv) {                              // the row's ragged end
                const float* p = row + 4 * v;
                x[u].x = __ldcg(p);
                x[u].y = 4 * v + 1 < n ? __ldcg(p + 1) : 0.f;
                x[u].z = 4 * v + 2 < n ? __ldcg(p + 2) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kSelUnroll; ++u) {
            const int j = 4 * (base + u * nt + tid);
            f(j + 0, float_key(__float_as_uint(x[u].x)), j + 0 < n);
            f(j + 1, float_key(__float_as_uint(x[u].y)), j + 1 < n);
            f(j + 2, float_key(__float_as_uint(x[u].z)), j + 2 < n);
            f(j + 3, float_key(__float_as_uint(x[u].w)), j + 3 < n);
        }
    }
}

// The same over a cached row in shared memory.
template <class F>
__device__ __forceinline__ void sel_cached_row(const uint32_t* kc, int n, F&& f)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int base = 0; base < n; base += nt) {
        const int j = base + tid;
        f(j, j < n ? kc[j] : 0u, j < n);
    }
}

// Selects the k largest of row[0 : n) (n > k >= 1) into out[0 : k) (any order).
// dyn: dyn_bytes of free shared memory (16-byte aligned) for the candidate
// store and the key cache.  The row must be 16-byte aligned.  Every thread of
// the block calls it; it ends with a block barrier.
static __device__ __noinline__ void select_row_cta(const float* __restrict__ row, int n, int k,
                                                   int32_t* __restrict__ out, SelectSmem& sh, uint8_t* dyn,
                                                   uint32_t dyn_bytes)
{
    const int tid = threadIdx.x, lane = tid & 31, nt = blockDim.x;
    const bool cached = static_cast<uint64_t>(n) * 4 + static_cast<uint64_t>(kSelCandCached) * 8 <= dyn_bytes;
    const int cand_cap = cached ? kSelCandCached : min(kSelCandMax, static_cast<int>(dyn_bytes / 8));
    uint32_t* ck = reinterpret_cast<uint32_t*>(dyn);
    int* cp = reinterpret_cast<int*>(dyn + 4 * cand_cap);
    uint32_t* kc = reinterpret_cast<uint32_t*>(dyn + 8 * cand_cap);

    for (int j = tid; j < kSelBins; j += nt)
        sh.hist[j] = 0;
    __syncthreads();

    // ---- 1. one pass: histogram of the top 11 key bits (and the key cache)
    sel_stream_row(row, n, [&](int j, uint32_t key, bool valid) {
        if (valid) {
            if (cached)
                kc[j] = key;
            atomicAdd(&sh.hist[key >> 21], 1);
        }
    });
    __syncthreads();
    sel_find_bin(sh, sh.hist, kSelBins, k);
    int need = k - sh.above;
    int in_bin = sh.in_bin;
    uint32_t lo = static_cast<uint32_t>(sh.bin) << 21, hi = lo + ((1u << 21) - 1u);
    __syncthreads();

    // ---- 2. refine the threshold bin while it overflows the candidate store
    int shift = 21;
    while (in_bin > cand_cap && shift > 0) {
        shift = max(0, sel_log2_ceil(static_cast<uint64_t>(hi) - lo + 1) - kSelBinBits);
        for (int j = tid; j < kSelBins; j += nt)
            sh.hist[j] = 0;
        __syncthreads();
        auto count = [&](int, uint32_t key, bool valid) {
            if (valid && key >= lo && key <= hi)
                atomicAdd(&sh.hist[(key - lo) >> shift], 1);
        };
        if (cached)
            sel_cached_row(kc, n, count);
        else
            sel_stream_row(row, n, count);
        __syncthreads();
        sel_find_bin(sh, sh.hist, kSelBins, need);
        need -= sh.above;
        in_bin = sh.in_bin;
        const uint32_t blo = lo + (static_cast<uint32_t>(sh.bin) << shift);
        hi = static_cast<uint32_t>(
            min(static_cast<uint64_t>(hi), static_cast<uint64_t>(blo) + ((uint64_t(1) << shift) - 1)));
        lo = blo;
        __syncthreads();
    }
    const int n_direct = k - need;                 // keys > hi, all taken

    // ---- 3. output pass: keys above the bin out, the bin's keys to the
    // candidates.  Each thread counts its own keys, one block scan gives every
    // thread its output and candidate offsets, and a second sweep writes them:
    // no shared counter is contended.
    int n_up = 0, n_cd = 0;
    auto count = [&](int, uint32_t key, bool valid) {
        n_up += (valid && key > hi) ? 1 : 0;
        n_cd += (valid && key >= lo && key <= hi) ? 1 : 0;
    };
    if (cached) {
        for (int j = tid; j < n; j += nt)          // strided: conflict-free shared loads
            count(j, kc[j], true);
    } else {
        sel_stream_row(row, n, count);
    }
    int off_up, off_cd;
    {
        int tot;
        if (n < 65536) {                           // both counts in one scan
            const int v = n_up | (n_cd << 16);
            const uint32_t ex = static_cast<uint32_t>(sel_block_scan(v, sh.ws, &tot) - v);
            off_up = static_cast<int>(ex & 0xFFFFu);
            off_cd = static_cast<int>(ex >> 16);
            if (tid == 0)
                sh.ncand = static_cast<int>(static_cast<uint32_t>(tot) >> 16);
        } else {
            off_up = sel_block_scan(n_up, sh.ws, &tot) - n_up;
            off_cd = sel_block_scan(n_cd, sh.ws, &tot) - n_cd;
            if (tid == 0)
                sh.ncand = tot;
        }
    }
    auto write = [&](int j, uint32_t key, bool valid) {
        if (valid && key > hi) {
            out[off_up++] = j;
        } else if (valid && key >= lo) {
            if (off_cd < cand_cap) {
                ck[off_cd] = key;
                cp[off_cd] = j;
            }
            ++off_cd;
        }
    };
    if (cached) {
        for (int j = tid; j < n; j += nt)
            write(j, kc[j], true);
    } else {
        sel_stream_row(row, n, write);
    }
    __syncthreads();

    // ---- 4. the `need` best candidates by (key desc, position asc)
    const int cand_total = sh.ncand;
    auto cand_order = [&](int j) -> uint64_t {
        return (static_cast<uint64_t>(ck[j] - lo) << 32) |
               static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(cp[j]));
    };
    if (cand_total == need && cand_total <= cand_cap) {
        for (int t = tid; t < cand_total; t += nt)
            out[n_direct + t] = cp[t];
    } else if (cand_total <= kSelRankMax) {
        for (int t = tid; t < cand_total; t += nt) {
            const uint64_t ot = cand_order(t);
            int rank = 0;
            for (int j = 0; j < cand_total; ++j)
                rank += cand_order(j) > ot ? 1 : 0;
            if (rank < need)
                out[n_direct + rank] = cp[t];
        }
    } else if (cand_total <= cand_cap) {
        // radix selection, 8-bit digits from the top of the 64-bit order; it stops
        // as soon as the chosen digit's bin holds exactly the number still needed
        int* h8 = sh.hist;                         // 256 bins
        const int key_bits = sel_log2_ceil(static_cast<uint64_t>(hi - lo) + 1);
        uint64_t prefix = 0;
        int rem = need;
        int top = 32 + key_bits;                   // bits [0, top) still undecided
        while (top > 0) {
            const int lo_bit = max(0, top - 8);
            const uint64_t mask = (uint64_t(1) << (top - lo_bit)) - 1;
            if (tid < 256)
                h8[tid] = 0;
            __syncthreads();
            for (int j = tid; j < cand_total; j += nt) {
                const uint64_t o = cand_order(j);
                if (top >= 64 || (o >> top) == (prefix >> top))
                    atomicAdd(&h8[(o >> lo_bit) & mask], 1);
            }
            __syncthreads();
            sel_find_bin(sh, h8, 256, rem);
            prefix |= static_cast<uint64_t>(sh.bin) << lo_bit;
            rem -= sh.above;
            const int digit_in_bin = sh.in_bin;
            top = lo_bit;
            __syncthreads();
            if (digit_in_bin == rem)
                break;                             // the whole digit bin is taken
        }
        if (tid == 0)
            sh.nout = n_direct;
        __syncthreads();
        for (int base = 0; base < cand_total; base += nt) {
            const int j = base + tid;
            const bool t = j < cand_total && (top >= 64 ? true : (cand_order(j) >> top) >= (prefix >> top));
            const unsigned m = __ballot_sync(0xffffffffu, t);
            int slot = 0;
            if (lane == 0 && m)
                slot = atomicAdd(&sh.nout, __popc(m));
            slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(m & ((1u << lane) - 1u));
            if (t)
                out[slot] = cp[j];
        }
    } else {
        // one key value (the bin narrowed to a single key) held by more keys than
        // the candidate store: the `need` lowest positions holding it, in order
        const uint32_t key_eq = lo;
        int seen = 0;
        for (int base = 0; base < n && seen < need; base += nt) {
            const int s = base + tid;
            uint32_t key = 0;
            if (s < n)
                key = cached ? kc[s] : float_key(__float_as_uint(__ldcg(row + s)));
            const int is_eq = (s < n && key == key_eq) ? 1 : 0;
            int tot;
            const int incl = sel_block_scan(is_eq, sh.ws, &tot);
            const int rank = seen + incl - 1;
            if (is_eq && rank < need)
                out[n_direct + rank] = s;
            seen += tot;
        }
    }
    __syncthreads();
}

// Short rows: every visible position, then -1 padding.
__device__ __forceinline__ void select_short_row_cta(int n, int k, int32_t* __restrict__ out)
{
    for (int s = threadIdx.x; s < k; s += blockDim.x)
        out[s] = s < n ? s : -1;
}

}  // namespace dsa
