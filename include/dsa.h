/*
 * dsa.h -- C ABI of libdsa, the GB300 (sm_103a) DeepSeek sparse-attention
 * decode path: paged lightning-indexer MQA logits, per-row top-k, sparse MLA
 * decode, and a device-side schedule builder for CUDA-graph capture.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or retains them past the call.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *    void*, NULL = legacy default stream).  No entry point synchronises or reads
 *    device memory from the host, except dsa_get_device_status().  Every
 *    compute entry point may therefore be captured into a CUDA graph.
 *  - Strides are in BYTES unless stated otherwise.
 *  - Arguments are validated on the host before anything is enqueued; an
 *    invalid call returns an error code and enqueues nothing.  Conditions that
 *    only the device can see (a block-table entry out of range, a visible
 *    length above the logits width, an index outside the block table) make the
 *    kernel skip the offending access and OR a bit into the caller's int32
 *    status word `status_dev` (nullable = not reported).
 *  - The library is stateless apart from a per-thread record of the last CUDA
 *    error (dsa_last_cuda_error) and is safe to call from several threads.
 *
 * Sources: "SM120 FP8 paged MQA page 32" (vllm-project/DeepGEMM #14), Summary:
 * FP8 paged MQA logits with block_kv 32/64, next_n >= 1, varlen; "feat(deepseek_v4):
 * Add fp4 indexer for dsv4" (ROCm/ATOM #1709), commit notes: FP4 indexer,
 * indexer_score_topk, schedule built into a fixed-address CUDA-graph buffer,
 * prefill logits width and Q-row budget chunking; "Add DeepSeek V4 sparse MLA
 * TRTLLM-GEN kernels" (flashinfer #3269): sparse MLA decode over top-k indices.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride / alignment */
    DSA_ERR_UNSUPPORTED = 2, /* shape or format this build has no kernel for; wrong GPU arch */
    DSA_ERR_CAPACITY = 3,    /* a caller buffer (schedule, workspace) is too small */
    DSA_ERR_CUDA = 4         /* a CUDA call failed; see dsa_last_cuda_error() */
} dsa_status;

/* Storage formats of a paged cache. */
typedef enum {
    DSA_KV_FP8_E4M3 = 0, /* e4m3 values + one fp32 scale per token */
    DSA_KV_MXFP4 = 1,    /* packed e2m1 values (even element in the low nibble) +
                            one ue8m0 scale per 32 elements */
    DSA_KV_BF16 = 2      /* bf16 values, no scale */
} dsa_format;

/* Element types of unquantised inputs. */
#define DSA_DTYPE_F32 0
#define DSA_DTYPE_BF16 1

/* Bits OR-ed into the caller's device status word. */
#define DSA_DEV_BAD_PAGE 0x1  /* block_table entry outside [0, num_pages): access skipped */
#define DSA_DEV_WIDTH 0x2     /* visible length > logits_width: clipped to the width */
#define DSA_DEV_TIMEOUT 0x4   /* a bounded on-chip wait gave up; outputs are invalid */
#define DSA_DEV_BAD_INDEX 0x8 /* top-k index beyond the block table: token skipped */
#define DSA_DEV_SCHEDULE 0x10 /* schedule buffer does not describe this call */

/*
 * One paged cache.  Token t (0 <= t < page_kv) of physical page p has its
 * values at  values + p*val_page_stride + t*val_token_stride  and its scales at
 * scales + p*sc_page_stride + t*sc_token_stride.  Logical token s of sequence b
 * lives in physical page block_table[b*bt_row_stride + s/page_kv], row s%page_kv
 * (the paged layout of "SM120 FP8 paged MQA page 32", Summary: shuffled physical
 * pages, padded page strides).  Values and scales may share one allocation
 * (the "fused" cache: scales after the page's values).
 *
 * Alignment required by the tensor-memory-access (TMA) paths: values, scales
 * and the page strides 16-byte aligned; val_token_stride == the dense row size
 * (head_dim bytes for FP8, head_dim/2 for MXFP4, 2*head_dim for BF16);
 * sc_token_stride == 4 (FP8) or head_dim/32 (MXFP4).
 *
 * Compressed indexer caches ("feat(deepseek_v4): Add fp4 indexer for dsv4":
 * the CSA index length is context_len // 4; "SM120 FP8 paged MQA page 32":
 * a 64-token storage block holds 32 states of a ratio-2 layer): with
 * compress_ratio = c > 1, entry e of a sequence summarises tokens
 * [c*e, c*e + c), the block table addresses ENTRIES (page_kv entries per
 * page), and a row that sees vis tokens sees floor(vis / c) entries; logits
 * and top-k positions are entry indices.  Layers of different ratios can share
 * one block table and physical pool, each with its own page_kv.  1 <= c <= 65536.
 */
typedef struct {
    int32_t fmt;               /* dsa_format */
    int32_t head_dim;          /* elements per token */
    int32_t page_kv;           /* tokens per page: 32 or 64 */
    int32_t num_pages;         /* pages in the pool */
    const void* values;        /* device */
    int64_t val_page_stride;   /* bytes */
    int64_t val_token_stride;  /* bytes */
    const void* scales;        /* device; NULL for BF16 */
    int64_t sc_page_stride;    /* bytes */
    int64_t sc_token_stride;   /* bytes */
    const int32_t* block_table; /* device, [batch, bt_row_stride] int32 */
    int64_t bt_row_stride;     /* ELEMENTS between sequences' rows */
    int32_t max_pages_per_seq; /* valid columns of each block-table row */
    int32_t compress_ratio;    /* indexer caches: tokens per entry (0 or 1: one
                                  entry per token); see below */
} dsa_paged_cache;

/* Human-readable name of a status code (static string, never NULL). */
DSA_API const char* dsa_status_string(dsa_status status);

/* cudaError_t of the last failed CUDA call made by this thread (0 = none). */
DSA_API int dsa_last_cuda_error(void);

/* Library ABI version (major*100 + minor).  1.01: indexer_mqa_logits_paged
 * accepts sched = NULL for calls of at most 256 work units.  1.02: fused
 * indexer_score_topk, dsa_kv_quantize_scatter, dsa_wait_selftest.  2.00:
 * compressed indexer caches (dsa_paged_cache.compress_ratio; a compress_ratio
 * argument of dsa_indexer_build_schedule and indexer_topk),
 * sparse_mla_decode_swa, MLA caches of any page size. */
DSA_API int dsa_version(void);

/*
 * Indexer schedule ("feat(deepseek_v4): Add fp4 indexer for dsv4", commit notes:
 * the decode schedule is built by one kernel straight into a fixed-address
 * CUDA-graph buffer and the logits kernel then skips its own build; cta_info
 * holds absolute row ids, so each prefill chunk needs its own schedule).
 *
 * The rows [row_begin, row_end) of a batch (row r = sequence r/next_n, draft
 * position r%next_n) are grouped into work units of at most
 * max(1, min(next_n, 256/num_heads)) consecutive rows of one sequence; each unit
 * is split into 128-token tiles up to the largest visible length of its rows.
 * dsa_indexer_schedule_bytes() gives the buffer size for a call shape (it
 * depends only on host-known values); dsa_indexer_build_schedule() fills it on
 * the device from the device-resident context_lens, so the buffer can be built
 * inside a captured graph at every replay.
 *
 * context_lens: device int32 [batch], lengths INCLUDING the next_n new tokens.
 * compress_ratio: the K cache's compress_ratio (0 or 1: one entry per token).
 * sched: device buffer of at least dsa_indexer_schedule_bytes(...) bytes,
 *        16-byte aligned, caller-owned; its contents are opaque.
 * Errors: DSA_ERR_INVALID_ARG (sizes, row range, null pointers),
 *         DSA_ERR_CAPACITY (sched_bytes too small).
 */
DSA_API size_t dsa_indexer_schedule_bytes(int batch, int next_n, int num_heads, int row_begin,
                                  int row_end);
DSA_API dsa_status dsa_indexer_build_schedule(const int32_t* context_lens, int batch, int next_n,
                                      int num_heads, int compress_ratio, int row_begin,
                                      int row_end, void* sched, size_t sched_bytes,
                                      int32_t* status_dev, void* stream);

/*
 * Paged lightning-indexer MQA logits (DeepSeek sparse attention):
 *   logits[r - row_begin][s] = k_scale[s] * sum_h w[r][h] * relu(sum_d q[r][h][d] * k[s][d])
 * for row_begin <= r < row_end and 0 <= s < vis(r), where for sequence
 * b = r/next_n, draft position i = r%next_n and L = context_lens[b]:
 *   vis(r) = clamp(L - next_n + i + 1, 0, L)
 * (next_n = 1: all L tokens; a causal prefill is batch 1, next_n = L).
 * Entries at s >= vis(r) are left untouched.
 *
 * q:        FP8:   [rows_total, num_heads, head_dim] e4m3 bytes (absolute rows).
 *           MXFP4: [rows_total, num_heads, head_dim/2] packed e2m1, with
 * q_scales: [rows_total, num_heads, head_dim/32] ue8m0 (MXFP4 only, else NULL).
 * q_fmt:    must equal k->fmt (DSA_KV_FP8_E4M3 or DSA_KV_MXFP4).
 * weights:  fp32 [rows_total, num_heads], 16-byte aligned.
 * k:        the paged indexer K cache; FP8 caches carry k_scale per token,
 *           MXFP4 caches carry block scales only (k_scale = 1).
 * sched:    built by dsa_indexer_build_schedule() with the same batch, next_n,
 *           num_heads, row_begin, row_end (and current context_lens); or NULL
 *           (sched_bytes ignored) for calls of at most 256 work units, whose
 *           units the kernel then builds itself from context_lens (one launch
 *           instead of two; larger calls without a schedule get DSA_ERR_CAPACITY).
 * logits:   fp32, row (r - row_begin) at logits + (r-row_begin)*logits_row_stride
 *           (ELEMENTS); logits_width = columns available per row.  A decode
 *           step under graph capture keeps a fixed width; a prefill sizes it to
 *           the actual longest visible length ("Add fp4 indexer for dsv4",
 *           prefill logits width note).
 * Supported: head_dim in {32, 64, 128} (FP8) or {64, 128} (MXFP4); num_heads in
 *           {4, 8, 16, 32, 64, 128}; page_kv in {32, 64}.  MXFP4 at head_dim 128
 *           also needs min(next_n, 256/num_heads) * num_heads <= 128.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (sched_bytes), CUDA.
 */
DSA_API dsa_status indexer_mqa_logits_paged(const void* q, const void* q_scales, int q_fmt,
                                    const float* weights, int num_heads,
                                    const dsa_paged_cache* k, const int32_t* context_lens,
                                    int batch, int next_n, int row_begin, int row_end,
                                    const void* sched, size_t sched_bytes, float* logits,
                                    int64_t logits_row_stride, int logits_width,
                                    int32_t* status_dev, void* stream);

/*
 * Fused indexer score + top-k ("feat(deepseek_v4): Add fp4 indexer for dsv4",
 * commit notes: indexer_score_topk scores the paged K cache and returns each
 * row's top-k token positions in one op).  Computes exactly what
 * indexer_mqa_logits_paged() followed by indexer_topk() compute -- the same
 * logits in `logits`, the same index sets in idx / count -- in ONE launch: the
 * block that scores a work unit's last outstanding tiles selects that unit's
 * rows from the logits just written, while the other blocks keep scoring.
 *
 * Arguments as indexer_mqa_logits_paged() (with logits 16-byte aligned and
 * logits_row_stride a multiple of 4) plus:
 * topk:     k, 1 <= k <= 16384.
 * idx:      int32 [rows, idx_row_stride >= k] (ELEMENTS), row r - row_begin:
 *           the positions of the row's min(k, vis) largest logits (any order;
 *           among equal logits the lower position wins), then -1.
 * count:    nullable int32 [rows]: min(k, vis).
 * workspace: device buffer of dsa_score_topk_workspace_bytes(...) bytes, 4-byte
 *           aligned, ALL ZERO before the first call (e.g. cudaMemset once after
 *           allocating it).  Every call that completes leaves it zero again, so
 *           it can be reused by the next call (and by graph replays) without
 *           clearing; after a call that reported DSA_DEV_TIMEOUT it must be
 *           cleared again.  Calls that overlap on the GPU need separate
 *           workspaces.
 * Errors: as indexer_mqa_logits_paged(); UNSUPPORTED (k); INVALID_ARG (idx,
 *         idx_row_stride, workspace); CAPACITY (ws_bytes).
 */
DSA_API size_t dsa_score_topk_workspace_bytes(int batch, int next_n, int num_heads, int row_begin,
                                              int row_end);
DSA_API dsa_status indexer_score_topk(const void* q, const void* q_scales, int q_fmt,
                                      const float* weights, int num_heads, const dsa_paged_cache* k,
                                      const int32_t* context_lens, int batch, int next_n,
                                      int row_begin, int row_end, const void* sched,
                                      size_t sched_bytes, float* logits, int64_t logits_row_stride,
                                      int logits_width, int topk, int32_t* idx,
                                      int64_t idx_row_stride, int32_t* count, void* workspace,
                                      size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Allocation-free variant of indexer_mqa_logits_paged() (no counterpart on the
 * pages; it exists for callers of this library that cannot allocate device
 * memory -- e.g. a plugin running under a host framework that owns the device
 * allocator and offers no hook, or a serving path that forbids cudaMalloc
 * while handling requests).
 *
 * Same arguments, operation, outputs and errors as indexer_mqa_logits_paged(),
 * minus the schedule buffer: the schedule is built into a fixed 256 KiB array
 * inside the library (one per GPU the process uses, held until exit), then the
 * logits kernel runs on it -- two launches on `stream`, nothing allocated.
 *  - Limit: at most 8191 work units (units = sequences for decode with
 *    next_n * num_heads <= 256; ceil(rows / (256 / num_heads)) for prefill);
 *    larger calls return DSA_ERR_CAPACITY and enqueue nothing.
 *  - The first call on a device looks up the array's device address (once per
 *    device and CUDA context, with that device current; again after a device
 *    reset); make that first call before any stream capture.
 *  - Every host check of indexer_mqa_logits_paged() runs before anything is
 *    enqueued, so a rejected call leaves the array as it was.
 *  - All calls share the one array: calls whose work overlaps on the GPU (other
 *    streams, other host threads) race on it and must be serialised by the
 *    caller.  Nothing needs clearing between calls: each call rewrites every
 *    schedule word it later reads.
 */
DSA_API dsa_status indexer_mqa_logits_paged_noalloc(const void* q, const void* q_scales, int q_fmt,
                                                    const float* weights, int num_heads,
                                                    const dsa_paged_cache* k,
                                                    const int32_t* context_lens, int batch,
                                                    int next_n, int row_begin, int row_end,
                                                    float* logits, int64_t logits_row_stride,
                                                    int logits_width, int32_t* status_dev,
                                                    void* stream);

/*
 * Per-row top-k of the indexer logits ("feat(deepseek_v4): Add fp4 indexer for
 * dsv4": indexer_score_topk; "Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels":
 * dynamic per-row top-k lengths).  For each row, the k largest of
 * logits[row][0 : vis(row)) (vis as above, clipped to logits_width) are
 * selected (vis in entries: floor(vis / compress_ratio), compress_ratio 0 or 1
 * meaning one entry per token); idx[row][0 : min(k, vis)) receives their
 * positions (in no particular order) and idx[row][min(k, vis) : k) receives -1.  Among exactly
 * equal logits (-0 equals +0) the lower position wins.  count (nullable)
 * receives min(k, vis).
 *
 * logits:   as produced by indexer_mqa_logits_paged (row stride in ELEMENTS).
 * idx:      int32 [rows, idx_row_stride >= k] (stride in ELEMENTS).
 * workspace: device scratch of dsa_topk_workspace_bytes(...) bytes (may be 0,
 *           then workspace may be NULL).
 * Supported: 1 <= k <= 16384.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (workspace), CUDA.
 */
DSA_API size_t dsa_topk_workspace_bytes(int rows, int logits_width, int k);
DSA_API dsa_status indexer_topk(const float* logits, int64_t logits_row_stride, int logits_width,
                        const int32_t* context_lens, int batch, int next_n, int compress_ratio,
                        int row_begin, int row_end, int k, int32_t* idx, int64_t idx_row_stride,
                        int32_t* count, void* workspace, size_t ws_bytes, int32_t* status_dev,
                        void* stream);

/*
 * Sparse MLA decode ("Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels":
 * trtllm_batch_decode_sparse_mla over top-k selected latent tokens, bf16 output
 * + LSE).  For row r (sequence b = seq_of_row ? seq_of_row[r] : r/next_n) and
 * head h, over the valid entries j (idx[r][j] >= 0) with latent rows
 * c_j = decode(latent[b][idx[r][j]]) * token_scale:
 *   s_j = softmax_scale * sum_{d < d_qk} q[r][h][d] * c_j[d]
 *   lse[r][h] = ln sum_j exp(s_j)                 (natural log)
 *   out[r][h][e] = sum_j exp(s_j - lse) * c_j[e]  for e < d_v
 * A row with no valid index gets out = 0 and lse = -inf.
 *
 * q_bf16:   bf16 [rows, num_heads, d_qk].
 * kv:       the paged latent cache (FP8 + fp32 token scale, or BF16) with
 *           head_dim == d_qk and any page_kv >= 1; the value vector is its
 *           first d_v elements.
 * idx:      int32 [rows, idx_row_stride >= k] (ELEMENTS), logical positions.
 * out_bf16: bf16 [rows, num_heads, d_v]; lse: fp32 [rows, num_heads].
 * workspace: device scratch of dsa_sparse_mla_workspace_bytes(...) bytes.
 * Supported: d_v <= d_qk <= 1024, d_qk % 16 == 0, d_v % 16 == 0.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (workspace), CUDA.
 */
DSA_API size_t dsa_sparse_mla_workspace_bytes(int rows, int num_heads, int d_qk, int d_v, int k);
DSA_API dsa_status sparse_mla_decode(const void* q_bf16, int rows, int num_heads, int d_qk, int d_v,
                             float softmax_scale, const dsa_paged_cache* kv,
                             const int32_t* seq_of_row, int next_n, const int32_t* idx,
                             int64_t idx_row_stride, int k, void* out_bf16, float* lse,
                             void* workspace, size_t ws_bytes, int32_t* status_dev,
                             void* stream);

/*
 * K-cache quantise / scatter ("feat(deepseek_v4): Add fp4 indexer for dsv4",
 * commit notes: the FP4 indexer's scatter kernel beside its mqa-logits kernel,
 * writing new tokens' K into the paged cache).  Token t's row of new K is
 * quantised and written to physical slot s = slot_mapping[t] of `cache`, i.e.
 * page s / page_kv, row s % page_kv (slots < 0 are padding and skipped; a page
 * >= num_pages sets DSA_DEV_BAD_PAGE and the token is skipped):
 *  - DSA_KV_FP8_E4M3: scale = amax / 448 over the token's head_dim values (fp32
 *    division; 1 for an all-zero row), codes e4m3(x / scale) (fp32 division,
 *    round to nearest, ties to even, saturating at +-448); the fp32 scale is
 *    stored at the token's scale slot.
 *  - DSA_KV_MXFP4 (OCP MX v1.0): per 32-element block, e = floor(log2 amax) - 2
 *    clamped to [-127, 127] (-127 for a zero block) stored as the ue8m0 byte
 *    e + 127, codes e2m1(x * 2^-e) (ties to even, saturating at +-6), two per
 *    byte with the even element in the low nibble.
 * The sign bit of every code is the sign bit of the value it encodes.
 *
 * k_new:    [n_tokens, k_row_stride] fp32 (k_dtype DSA_DTYPE_F32) or bf16
 *           (DSA_DTYPE_BF16); 16-byte aligned, row stride in ELEMENTS with
 *           stride * element size a multiple of 16.
 * slot_mapping: device int64 [n_tokens].
 * cache:    FP8 (head_dim % 8 == 0) or MXFP4 (head_dim % 32 == 0), head_dim <=
 *           4096; its values and scales are WRITTEN (only the addressed token
 *           rows); block_table is not used.  FP8: values 8-byte aligned, value
 *           strides multiples of 8, scale strides multiples of 4.  MXFP4: value
 *           strides multiples of 4.  Two tokens mapped to one slot race.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
DSA_API dsa_status dsa_kv_quantize_scatter(const void* k_new, int k_dtype, int64_t k_row_stride,
                                           int n_tokens, const int64_t* slot_mapping,
                                           const dsa_paged_cache* cache, int32_t* status_dev,
                                           void* stream);

/*
 * Self-test of the bounded waits (no counterpart on the pages; it checks a
 * property of this library).  Every on-chip wait in libdsa's kernels gives up
 * after a time limit and reports DSA_DEV_TIMEOUT instead of hanging.  This call
 * runs the same wait on a condition the caller controls: one thread waits, at
 * most limit_us microseconds, on a barrier that is arrived on only if
 * *flag == expect when the kernel reads it.  If the wait runs out it ORs
 * DSA_DEV_TIMEOUT into *status_dev and the kernel returns normally.
 * flag, status_dev: device int32 words.  1 <= limit_us <= 2,000,000.
 * Errors: INVALID_ARG, UNSUPPORTED (wrong GPU), CUDA.
 */
DSA_API dsa_status dsa_wait_selftest(const int32_t* flag, int32_t expect, int limit_us,
                                     int32_t* status_dev, void* stream);

/*
 * Sparse MLA decode over a sliding window plus selected entries ("Add DeepSeek
 * V4 sparse MLA TRTLLM-GEN kernels": trtllm_batch_decode_sparse_mla_dsv4 with
 * sliding_window_kv_cache, dynamic per-row sparse_topk_lens and varlen q
 * through cum_seq_lens_q).  Row r belongs to sequence b with query position i
 * and query length q_len: rows [cum_seq_lens_q[b], cum_seq_lens_q[b+1]) are
 * sequence b's (i = r - cum[b]); without cum_seq_lens_q, b = r / next_n,
 * i = r % next_n, q_len = next_n.  Its keys, in ONE softmax:
 *  - the first min(k, topk_lens[r]) entries of idx[r] that are >= 0 (all k
 *    when topk_lens is NULL): logical entries of sequence b in `kv`;
 *  - when swa is not NULL, the last w = min(window, vis) positions
 *    [vis - w, vis) of sequence b in `swa`, where
 *    vis = clamp(seq_lens[b] - q_len + i + 1, 0, seq_lens[b]) (the row's
 *    causal view of its sequence, seq_lens counting the new tokens).
 * Then as sparse_mla_decode(): s_j = softmax_scale * q . c_j[0:d_qk],
 * lse = ln sum_j exp(s_j), out = sum_j exp(s_j - lse) * c_j[0:d_v]; a row with
 * no key gets out = 0, lse = -inf (a row outside every sequence also sets
 * DSA_DEV_BAD_INDEX).
 *
 * kv, swa:  latent caches of the same format (FP8 + token scale, or BF16) with
 *           head_dim == d_qk and any page_kv >= 1 (a compressed cache may hold
 *           a few entries per physical block), each with its own block table.
 * topk_lens: nullable device int32 [rows].   seq_lens: device int32 [batch]
 *           (required with swa).   cum_seq_lens_q: nullable device int32
 *           [batch + 1], non-decreasing, cum[0] = 0, cum[batch] = rows.
 * Other arguments as sparse_mla_decode().
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY, CUDA.
 */
DSA_API dsa_status sparse_mla_decode_swa(const void* q_bf16, int rows, int num_heads, int d_qk, int d_v,
                                         float softmax_scale, const dsa_paged_cache* kv,
                                         const int32_t* idx, int64_t idx_row_stride, int k,
                                         const int32_t* topk_lens, const dsa_paged_cache* swa,
                                         int window, const int32_t* seq_lens,
                                         const int32_t* cum_seq_lens_q, int batch, int next_n,
                                         void* out_bf16, float* lse, void* workspace,
                                         size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Opt-in, SYNCHRONISING read of a device status word: waits for `stream`,
 * copies *status_dev into *host_out.  Never called by the other entry points.
 */
DSA_API dsa_status dsa_get_device_status(const int32_t* status_dev, int32_t* host_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
