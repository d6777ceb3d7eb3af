// common.cuh -- definitions shared by the libdsa kernels and their host launchers.
#pragma once

#include <cstdint>

#include "../../include/dsa.h"

namespace dsa {

// Tokens scored per indexer tile: one tcgen05 M=128 accumulator (one TMEM lane
// per token).
constexpr int kTileTokens = 128;
// Largest MMA N (rows x heads per work unit).
constexpr int kMaxUnitCols = 256;
// Largest unit count for which a logits launch without a schedule buffer builds
// the unit records itself (in shared memory, in every CTA).
constexpr int kInlineUnits = 256;

// Visible length of draft row i of a sequence of context length L with next_n
// new tokens: clamp(L - next_n + i + 1, 0, L) ("SM120 FP8 paged MQA page 32",
// Summary: next_n 1/2/3 + varlen; the context length counts the new tokens).
__host__ __device__ __forceinline__ int visible_len(int L, int next_n, int i)
{
    long long v = static_cast<long long>(L) - next_n + i + 1;
    v = v < 0 ? 0 : v;
    return static_cast<int>(v > L ? L : v);
}

// Entries row i sees in a compressed K cache of `ratio` tokens per entry:
// floor(visible_len / ratio) ("feat(deepseek_v4): Add fp4 indexer for dsv4",
// the CSA index length context_len // 4); ratio 1 is one entry per token.
__host__ __device__ __forceinline__ int visible_entries(int L, int next_n, int i, int ratio)
{
    const int v = visible_len(L, next_n, i);
    return ratio == 1 ? v : v / ratio;          // no integer division for uncompressed caches
}

// Rows per work unit for a head count: as many draft rows of one sequence as
// fit in one MMA N dimension.
__host__ __device__ __forceinline__ int unit_rows(int next_n, int num_heads)
{
    int g = kMaxUnitCols / num_heads;
    g = g < 1 ? 1 : g;
    return g < next_n ? g : next_n;
}

// --------------------------------------------------------------- schedule
//
// Layout of the caller-owned schedule buffer (int32 words):
//   header[0..7]: magic, num_units, rows_per_unit, row_begin, row_end, next_n,
//                 total_tiles, compression ratio
//   units[num_units] (32-byte records): first_row (absolute), nrows, seq,
//                 tile_begin (prefix of 128-token tiles over the units),
//                 tile_end, vis_max (largest visible entry count of the
//                 unit's rows), ctx_len (the sequence's context length, >= 0), 0.
//                 A record is everything a kernel needs about its unit, read
//                 with one 32-byte load and no dependent lookups.
constexpr int32_t kSchedMagic = 0x44534132;  // "DSA2"
constexpr int kSchedHeaderWords = 8;

struct __align__(16) SchedUnit {
    int32_t first_row;
    int32_t nrows;
    int32_t seq;
    int32_t tile_begin;
    int32_t tile_end;
    int32_t vis_max;
    int32_t ctx_len;
    int32_t pad;
};

__host__ __device__ __forceinline__ int64_t sched_bytes_for_units(int64_t num_units)
{
    return static_cast<int64_t>(kSchedHeaderWords) * 4 + num_units * static_cast<int64_t>(sizeof(SchedUnit));
}

// Number of units covering rows [row_begin, row_end): per sequence, the rows it
// owns in the range, in groups of rows_per_unit.
__host__ __device__ __forceinline__ int64_t count_units(int batch, int next_n, int rows_per_unit,
                                                         int row_begin, int row_end)
{
    if (row_end <= row_begin)
        return 0;
    const int b0 = row_begin / next_n, b1 = (row_end - 1) / next_n;
    int64_t total = 0;
    // sequences strictly inside the range own next_n rows each
    for (int b = b0; b <= b1 && b < batch; ++b) {
        const int lo = b * next_n > row_begin ? b * next_n : row_begin;
        const int hi = (b + 1) * next_n < row_end ? (b + 1) * next_n : row_end;
        total += (hi - lo + rows_per_unit - 1) / rows_per_unit;
        if (b == b0 && b1 - b0 > 2) {
            // middle sequences are identical: skip ahead in O(1)
            const int full = b1 - b0 - 1;
            total += static_cast<int64_t>(full) * ((next_n + rows_per_unit - 1) / rows_per_unit);
            b = b1 - 1;
        }
    }
    return total;
}

// Unit u -> (sequence, first absolute row, rows) for rows [row_begin, row_end).
__device__ __forceinline__ void unit_rows_of(int u, int next_n, int G, int row_begin, int row_end,
                                             int* seq, int* first_row, int* nrows)
{
    const int b0 = row_begin / next_n;
    const int lo0 = row_begin;
    const int hi0 = min((b0 + 1) * next_n, row_end);
    const int u_first = (hi0 - lo0 + G - 1) / G;
    const int U = (next_n + G - 1) / G;  // units of a sequence fully inside the range
    int b, lo, hi, j;
    if (u < u_first) {
        b = b0;
        lo = lo0;
        hi = hi0;
        j = u;
    } else {
        b = b0 + 1 + (u - u_first) / U;
        j = (u - u_first) % U;
        lo = b * next_n;
        hi = min((b + 1) * next_n, row_end);
    }
    *seq = b;
    *first_row = lo + j * G;
    *nrows = min(G, hi - *first_row);
}

// --------------------------------------------------------- sparse MLA rows
//
// Token slots of a sparse MLA row: the kept entries of its index list first,
// then its sliding-window positions, tagged with this bit (positions < 2^30).
constexpr int32_t kSwaTag = 0x40000000;

// Sequence, query position and query length of MLA row r: through cumulative
// query lengths (rows [cum_q[b], cum_q[b+1]) belong to sequence b; -1 if r is
// in none), an explicit row -> sequence map, or r / next_n.
struct MlaRowSeq {
    int seq, i, q_len;
};
__device__ __forceinline__ MlaRowSeq mla_row_seq(int r, const int32_t* cum_q, int batch, const int32_t* seq_of_row,
                                                 int next_n)
{
    MlaRowSeq o;
    if (cum_q) {
        int lo = 0, hi = batch;                  // last b with cum_q[b] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum_q[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int c0 = cum_q[lo], c1 = lo < batch ? cum_q[lo + 1] : c0;
        if (lo >= batch || r >= c1) {
            o.seq = -1;
            o.i = 0;
            o.q_len = 0;
        } else {
            o.seq = lo;
            o.i = r - c0;
            o.q_len = c1 - c0;
        }
    } else if (seq_of_row) {
        o.seq = seq_of_row[r];
        o.i = 0;
        o.q_len = 1;
    } else {
        o.seq = r / next_n;
        o.i = r % next_n;
        o.q_len = next_n;
    }
    return o;
}

// Top-k outputs of a fused indexer score + top-k launch (k = 0: logits only).
struct FusedTopk {
    int k;
    int32_t* idx;           // [rows, idx_stride] int32, row r - row_begin
    int64_t idx_stride;     // elements
    int32_t* count;         // nullable, [rows]
    int32_t* counters;      // [num_units] int32 workspace: zero on entry, zero again on exit
};

// Order-preserving map of an fp32 bit pattern to uint32 (larger float -> larger
// key).  -0 is mapped like +0 so that equal values get equal keys.
__host__ __device__ __forceinline__ uint32_t float_key(uint32_t bits)
{
    bits = (bits == 0x80000000u) ? 0u : bits;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

}  // namespace dsa
