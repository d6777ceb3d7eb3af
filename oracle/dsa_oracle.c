/*
 * dsa_oracle.c -- plain, slow, fp64 CPU oracle for the DeepSeek sparse-attention
 * decode path: lightning-indexer MQA logits over a paged FP8 / MXFP4 K cache,
 * per-row top-k, and sparse MLA decode over the selected latent tokens.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant with the CUDA library: every format
 * is decoded here from its definition, every loop follows the definition of the
 * quantity it computes, and nothing is blocked, fused or reordered.
 *
 * Sources (titles of the pages the method is described on):
 *  - "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709): the indexer
 *    is an MQA-logits score over (q_fp8, weights) followed by a top-k
 *    ("indexer_score_topk"); FP4 (MXFP4) or FP8 K cache; paged block tables;
 *    varlen windows per draft row; prefill logits width = actual visible length.
 *  - "SM120 FP8 paged MQA page 32" (vllm-project/DeepGEMM #14), Summary and
 *    Validation: FP8 paged MQA logits with page 32/64, next_n 1/2/3 + varlen,
 *    shuffled physical pages, padded page strides, empty history, partial pages,
 *    float64 reference.
 *  - "Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels" (flashinfer #3269), API and
 *    review comments: sparse MLA decode over top-k selected latent tokens with
 *    dynamic top-k lengths, bf16 output + LSE.
 *  - The indexer score itself (DeepSeek sparse attention, lightning indexer):
 *        logit[r, s] = k_scale[s] * sum_h w[r, h] * relu( sum_d q[r, h, d] * k[s, d] )
 *
 * Readings taken where the pages are silent:
 *  - visible length of draft row i of a sequence with context length L and
 *    next_n rows: clamp(L - next_n + i + 1, 0, L) (context length includes the
 *    next_n new tokens, bound inclusive);
 *  - over a compressed K cache whose entry e summarises `ratio` consecutive
 *    tokens ("feat(deepseek_v4): Add fp4 indexer for dsv4": the CSA index
 *    length is context_len // 4), the row sees floor(visible length / ratio)
 *    entries (ratio 1: one entry per token);
 *  - entries at s >= visible length are not written;
 *  - e2m1 packing: the low nibble of a byte is the even element;
 *  - MXFP4 caches carry no per-token scale (k_scale = 1);
 *  - top-k order: logit descending, ties by ascending index; -1 padding;
 *  - LSE is the natural log; a row with no valid index gives out = 0, lse = -inf;
 *  - MLA value vector = first d_v dims of the latent row, key = first d_qk dims.
 *
 * Parity pins: every function here is pinned by the CPU tests under tests/
 * (library decode of all codes, hand-computed cases, torch fp64 einsum / dense
 * softmax attention on dequantised tensors, invariances, brute force).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_PAGE 2

/* ---------------------------------------------------------------- decoding */

/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities; S.1111.111 is NaN; exponent field 0 is subnormal. */
double dsa_oracle_e4m3(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* OCP FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no NaN /
 * infinity; exponent field 0 is subnormal (0 or 0.5). */
double dsa_oracle_e2m1(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int m = nibble & 0x1;
    double mag;
    if (e == 0)
        mag = ldexp((double)m / 2.0, 1 - 1);
    else
        mag = ldexp(1.0 + (double)m / 2.0, e - 1);
    return sign ? -mag : mag;
}

/* OCP UE8M0 block scale: unsigned 8-bit exponent, value 2^(code - 127); 0xFF is NaN. */
double dsa_oracle_ue8m0(uint8_t code)
{
    if (code == 0xFF)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double dsa_oracle_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------- visibility */

/* Draft row i (0 <= i < next_n) of a sequence whose context length L already
 * counts the next_n new tokens sees the first L - next_n + i + 1 tokens,
 * clamped to [0, L].  next_n = 1 gives L; a causal prefill (next_n = L) gives i + 1. */
int dsa_oracle_visible(int L, int next_n, int i)
{
    long v = (long)L - (long)next_n + (long)i + 1;
    if (v < 0)
        v = 0;
    if (v > L)
        v = L;
    return (int)v;
}

static float load_f32(const uint8_t* p)
{
    float f;
    memcpy(&f, p, sizeof f);
    return f;
}

/* Logical token s of sequence b -> physical page through the block table. */
static int page_of(const int32_t* block_table, int64_t bt_stride, int max_pages, int page_kv,
                   int num_pages, int b, int s, int* page)
{
    int lp = s / page_kv;
    if (lp >= max_pages)
        return ORACLE_ERR_PAGE;
    *page = block_table[(int64_t)b * bt_stride + lp];
    if (*page < 0 || *page >= num_pages)
        return ORACLE_ERR_PAGE;
    return ORACLE_OK;
}

/* ------------------------------------------------------ indexer logits FP8 */

/* q:        [rows_total, H, D] e4m3 bytes, row-major (absolute row ids)
 * w:        [rows_total, H] fp32
 * kvals:    paged e4m3 values; token s of page p starts at p*vps + (s%P)*vts bytes
 * kscales:  paged fp32 scales; at p*sps + (s%P)*sts bytes
 * out:      out[(r - row_begin) * out_stride + s] for s < visible length  */
int dsa_oracle_logits_fp8(const uint8_t* q, const float* w, int H, int D,
                          const uint8_t* kvals, int64_t vps, int64_t vts,
                          const uint8_t* kscales, int64_t sps, int64_t sts,
                          const int32_t* block_table, int64_t bt_stride, int max_pages,
                          int page_kv, int num_pages, const int32_t* context_lens, int batch,
                          int next_n, int ratio, int row_begin, int row_end, double* out,
                          int64_t out_stride, int out_width)
{
    double lut[256];
    int c, err = ORACLE_OK;
    long r;
    if (H <= 0 || D <= 0 || page_kv <= 0 || next_n <= 0 || ratio <= 0 || row_begin < 0 ||
        row_end > batch * next_n || row_begin > row_end)
        return ORACLE_ERR_ARG;
    for (c = 0; c < 256; ++c)
        lut[c] = dsa_oracle_e4m3((uint8_t)c);

#pragma omp parallel for schedule(dynamic, 1)
    for (r = row_begin; r < row_end; ++r) {
        int b = (int)(r / next_n), i = (int)(r % next_n);
        int vis = dsa_oracle_visible(context_lens[b], next_n, i) / ratio;
        int s;
        if (vis > out_width) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        for (s = 0; s < vis; ++s) {
            int page, h, d;
            const uint8_t* krow;
            double k_scale, acc = 0.0;
            if (page_of(block_table, bt_stride, max_pages, page_kv, num_pages, b, s, &page)) {
#pragma omp atomic write
                err = ORACLE_ERR_PAGE;
                break;
            }
            krow = kvals + (int64_t)page * vps + (int64_t)(s % page_kv) * vts;
            k_scale = (double)load_f32(kscales + (int64_t)page * sps + (int64_t)(s % page_kv) * sts);
            for (h = 0; h < H; ++h) {
                const uint8_t* qh = q + ((int64_t)r * H + h) * D;
                double dot = 0.0;
                for (d = 0; d < D; ++d)
                    dot += lut[qh[d]] * lut[krow[d]];
                acc += (double)w[(int64_t)r * H + h] * (dot > 0.0 ? dot : 0.0);
            }
            out[(r - row_begin) * out_stride + s] = k_scale * acc;
        }
    }
    return err;
}

/* ---------------------------------------------------- indexer logits MXFP4 */

/* Element d of a packed e2m1 row: byte d/2, low nibble for even d. */
static uint8_t e2m1_nibble(const uint8_t* row, int d)
{
    uint8_t byte = row[d / 2];
    return (d % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
}

/* q:        [rows_total, H, D/2] packed e2m1;  q_sc: [rows_total, H, D/32] ue8m0
 * kvals:    paged packed e2m1 rows (D/2 bytes), byte strides vps / vts
 * kscales:  paged ue8m0 rows (D/32 bytes), byte strides sps / sts
 * Each element is e2m1 * 2^(e - 127) of its 32-element block; no per-token scale. */
int dsa_oracle_logits_mxfp4(const uint8_t* q, const uint8_t* q_sc, const float* w, int H, int D,
                            const uint8_t* kvals, int64_t vps, int64_t vts,
                            const uint8_t* kscales, int64_t sps, int64_t sts,
                            const int32_t* block_table, int64_t bt_stride, int max_pages,
                            int page_kv, int num_pages, const int32_t* context_lens, int batch,
                            int next_n, int ratio, int row_begin, int row_end, double* out,
                            int64_t out_stride, int out_width)
{
    int err = ORACLE_OK;
    long r;
    if (H <= 0 || D <= 0 || D % 32 != 0 || page_kv <= 0 || next_n <= 0 || ratio <= 0 || row_begin < 0 ||
        row_end > batch * next_n || row_begin > row_end)
        return ORACLE_ERR_ARG;

#pragma omp parallel for schedule(dynamic, 1)
    for (r = row_begin; r < row_end; ++r) {
        int b = (int)(r / next_n), i = (int)(r % next_n);
        int vis = dsa_oracle_visible(context_lens[b], next_n, i) / ratio;
        int s;
        if (vis > out_width) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        for (s = 0; s < vis; ++s) {
            int page, h, d;
            const uint8_t *krow, *ksc;
            double acc = 0.0;
            if (page_of(block_table, bt_stride, max_pages, page_kv, num_pages, b, s, &page)) {
#pragma omp atomic write
                err = ORACLE_ERR_PAGE;
                break;
            }
            krow = kvals + (int64_t)page * vps + (int64_t)(s % page_kv) * vts;
            ksc = kscales + (int64_t)page * sps + (int64_t)(s % page_kv) * sts;
            for (h = 0; h < H; ++h) {
                const uint8_t* qh = q + ((int64_t)r * H + h) * (D / 2);
                const uint8_t* qs = q_sc + ((int64_t)r * H + h) * (D / 32);
                double dot = 0.0;
                for (d = 0; d < D; ++d) {
                    double qv = dsa_oracle_e2m1(e2m1_nibble(qh, d)) * dsa_oracle_ue8m0(qs[d / 32]);
                    double kv = dsa_oracle_e2m1(e2m1_nibble(krow, d)) * dsa_oracle_ue8m0(ksc[d / 32]);
                    dot += qv * kv;
                }
                acc += (double)w[(int64_t)r * H + h] * (dot > 0.0 ? dot : 0.0);
            }
            out[(r - row_begin) * out_stride + s] = acc;
        }
    }
    return err;
}

/* ------------------------------------------------------------------ top-k */

typedef struct {
    double v;
    int32_t s;
} scored;

/* Descending logit; equal logits by ascending token index. */
static int by_logit_desc(const void* a, const void* b)
{
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->s > y->s) - (x->s < y->s);
}

/* Full sort of each row's visible logits; the first min(k, vis) token indices are
 * written (in sorted order), the rest of the k slots get -1.  If count is not
 * NULL it receives min(k, vis) per row.  logits rows are chunk-relative
 * (row r at (r - row_begin) * stride). */
int dsa_oracle_topk(const double* logits, int64_t stride, const int32_t* context_lens, int batch,
                    int next_n, int ratio, int row_begin, int row_end, int k, int32_t* idx,
                    int64_t idx_stride, int32_t* count)
{
    long r;
    int err = ORACLE_OK;
    if (k <= 0 || next_n <= 0 || ratio <= 0 || row_begin < 0 || row_end > batch * next_n || row_begin > row_end)
        return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = row_begin; r < row_end; ++r) {
        int b = (int)(r / next_n), i = (int)(r % next_n);
        int vis = dsa_oracle_visible(context_lens[b], next_n, i) / ratio;
        int s, take = vis < k ? vis : k;
        int32_t* out = idx + (r - row_begin) * idx_stride;
        scored* buf = (scored*)malloc(sizeof(scored) * (size_t)(vis > 0 ? vis : 1));
        if (!buf) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        for (s = 0; s < vis; ++s) {
            buf[s].v = logits[(r - row_begin) * stride + s];
            buf[s].s = s;
        }
        qsort(buf, (size_t)vis, sizeof(scored), by_logit_desc);
        for (s = 0; s < k; ++s)
            out[s] = s < take ? buf[s].s : -1;
        if (count)
            count[r - row_begin] = take;
        free(buf);
    }
    return err;
}

/* -------------------------------------------------------- sparse MLA decode */

#define ORACLE_FMT_FP8 0
#define ORACLE_FMT_BF16 2

/* q:        [rows, Hq, d_qk] bf16 bits
 * latent:   paged rows of d_qk elements (e4m3 bytes + fp32 token scale, or bf16)
 * idx:      [rows, k] logical token indices of the row's sequence; < 0 = unused
 * For each (row, head): s_j = softmax_scale * q . c_j[0:d_qk] over valid j,
 *   lse = ln sum_j exp(s_j), out = sum_j exp(s_j - lse) * c_j[0:d_v].
 * No valid index: out = 0, lse = -inf. */
int dsa_oracle_sparse_mla(const uint16_t* q, int rows, int Hq, int d_qk, int d_v,
                          double softmax_scale, int fmt, const uint8_t* cvals, int64_t vps,
                          int64_t vts, const uint8_t* cscales, int64_t sps, int64_t sts,
                          const int32_t* block_table, int64_t bt_stride, int max_pages,
                          int page_kv, int num_pages, const int32_t* seq_of_row, int next_n,
                          const int32_t* idx, int64_t idx_stride, int k, double* out,
                          double* lse)
{
    int err = ORACLE_OK;
    long r;
    if (rows < 0 || Hq <= 0 || d_qk <= 0 || d_v <= 0 || d_v > d_qk || k < 0 || page_kv <= 0 ||
        (fmt != ORACLE_FMT_FP8 && fmt != ORACLE_FMT_BF16) || (!seq_of_row && next_n <= 0))
        return ORACLE_ERR_ARG;

#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < rows; ++r) {
        int b = seq_of_row ? seq_of_row[r] : (int)(r / next_n);
        int j, h, d, nvalid = 0;
        double* c = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)d_qk);
        double* sc = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
        if (!c || !sc) {
            free(c);
            free(sc);
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        /* dequantise the selected latent rows */
        for (j = 0; j < k; ++j) {
            int s = idx[r * idx_stride + j], page;
            const uint8_t* row;
            double tok_scale = 1.0;
            if (s < 0)
                continue;
            if (page_of(block_table, bt_stride, max_pages, page_kv, num_pages, b, s, &page)) {
#pragma omp atomic write
                err = ORACLE_ERR_PAGE;
                continue;
            }
            row = cvals + (int64_t)page * vps + (int64_t)(s % page_kv) * vts;
            if (fmt == ORACLE_FMT_FP8)
                tok_scale = (double)load_f32(cscales + (int64_t)page * sps + (int64_t)(s % page_kv) * sts);
            for (d = 0; d < d_qk; ++d) {
                double v;
                if (fmt == ORACLE_FMT_FP8) {
                    v = dsa_oracle_e4m3(row[d]) * tok_scale;
                } else {
                    uint16_t bits;
                    memcpy(&bits, row + 2 * d, 2);
                    v = dsa_oracle_bf16(bits);
                }
                c[(size_t)nvalid * d_qk + d] = v;
            }
            ++nvalid;
        }
        for (h = 0; h < Hq; ++h) {
            const uint16_t* qh = q + ((int64_t)r * Hq + h) * d_qk;
            double* o = out + ((int64_t)r * Hq + h) * d_v;
            double m = -INFINITY, l = 0.0, L;
            for (d = 0; d < d_v; ++d)
                o[d] = 0.0;
            if (nvalid == 0) {
                lse[(int64_t)r * Hq + h] = -INFINITY;
                continue;
            }
            for (j = 0; j < nvalid; ++j) {
                double dot = 0.0;
                for (d = 0; d < d_qk; ++d)
                    dot += dsa_oracle_bf16(qh[d]) * c[(size_t)j * d_qk + d];
                sc[j] = softmax_scale * dot;
                if (sc[j] > m)
                    m = sc[j];
            }
            for (j = 0; j < nvalid; ++j)
                l += exp(sc[j] - m);
            L = m + log(l);
            lse[(int64_t)r * Hq + h] = L;
            for (j = 0; j < nvalid; ++j) {
                double p = exp(sc[j] - L);
                for (d = 0; d < d_v; ++d)
                    o[d] += p * c[(size_t)j * d_qk + d];
            }
        }
        free(c);
        free(sc);
    }
    return err;
}

/* ------------------------------------ sparse MLA with a sliding window */

/* Latent row of logical position s of sequence b in a paged cache, decoded to
 * fp64 (e4m3 * token scale, or bf16) into c[0 : d).  Returns ORACLE_ERR_PAGE
 * if the block-table entry is missing or outside the pool. */
static int latent_row(int fmt, const uint8_t* vals, int64_t vps, int64_t vts, const uint8_t* scs, int64_t sps,
                      int64_t sts, const int32_t* bt, int64_t bt_stride, int max_pages, int page_kv, int num_pages,
                      int b, int s, int d, double* c)
{
    int page, e;
    const uint8_t* row;
    double tok_scale = 1.0;
    if (page_of(bt, bt_stride, max_pages, page_kv, num_pages, b, s, &page))
        return ORACLE_ERR_PAGE;
    row = vals + (int64_t)page * vps + (int64_t)(s % page_kv) * vts;
    if (fmt == 0)
        tok_scale = (double)load_f32(scs + (int64_t)page * sps + (int64_t)(s % page_kv) * sts);
    for (e = 0; e < d; ++e) {
        if (fmt == 0) {
            c[e] = dsa_oracle_e4m3(row[e]) * tok_scale;
        } else {
            uint16_t bits;
            memcpy(&bits, row + 2 * e, 2);
            c[e] = dsa_oracle_bf16(bits);
        }
    }
    return ORACLE_OK;
}

/* Sparse MLA decode over two latent caches in ONE softmax ("Add DeepSeek V4
 * sparse MLA TRTLLM-GEN kernels": sparse attention over the top-k selected
 * entries of one cache plus a sliding-window cache, dynamic per-row top-k
 * lengths, varlen q through cumulative query lengths).  For row r:
 *  - its sequence b and query position i: rows [cum_q[b], cum_q[b+1]) belong to
 *    sequence b (i = r - cum_q[b], q_len = cum_q[b+1] - cum_q[b]); without
 *    cum_q, b = r / next_n, i = r % next_n, q_len = next_n;
 *  - its visible length in the window cache's token stream:
 *    vis = clamp(seq_lens[b] - q_len + i + 1, 0, seq_lens[b]);
 *  - its keys: the first min(k, topk_lens[r]) entries of idx[r] that are >= 0
 *    (topk_lens NULL: all k), rows of the sparse cache; then the last
 *    min(window, vis) visible positions [vis - w, vis) of the window cache
 *    (none when wvals is NULL);
 *  - s_j = scale * q . c_j[0:d_qk], lse = ln sum_j exp(s_j),
 *    out = sum_j exp(s_j - lse) c_j[0:d_v]; no key: out = 0, lse = -inf.
 * Both caches have the format fmt (0 FP8 + token scale, 2 bf16). */
int dsa_oracle_sparse_mla_swa(const uint16_t* q, int rows, int Hq, int d_qk, int d_v, double softmax_scale,
                              int fmt, const uint8_t* cvals, int64_t vps, int64_t vts, const uint8_t* cscales,
                              int64_t sps, int64_t sts, const int32_t* bt, int64_t bt_stride, int max_pages,
                              int page_kv, int num_pages, const int32_t* idx, int64_t idx_stride, int k,
                              const int32_t* topk_lens, const uint8_t* wvals, int64_t wvps, int64_t wvts,
                              const uint8_t* wscales, int64_t wsps, int64_t wsts, const int32_t* wbt,
                              int64_t wbt_stride, int wmax_pages, int wpage_kv, int wnum_pages, int window,
                              const int32_t* seq_lens, const int32_t* cum_q, int batch, int next_n, double* out,
                              double* lse)
{
    int err = ORACLE_OK;
    long r;
    if (rows < 0 || Hq <= 0 || d_qk <= 0 || d_v <= 0 || d_v > d_qk || k < 0 || page_kv <= 0 || window < 0 ||
        (fmt != ORACLE_FMT_FP8 && fmt != ORACLE_FMT_BF16) || (!cum_q && next_n <= 0) || batch < 0 ||
        (wvals && wpage_kv <= 0))
        return ORACLE_ERR_ARG;

#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < rows; ++r) {
        int b, i, q_len, L, vis, kr, w, j, h, d, nkeys = 0;
        int maxkeys = k + (wvals ? window : 0);
        double *c, *sc;
        if (cum_q) {
            for (b = 0; b < batch; ++b)
                if (r >= cum_q[b] && r < cum_q[b + 1])
                    break;
            if (b == batch) {
#pragma omp atomic write
                err = ORACLE_ERR_ARG;
                continue;
            }
            i = (int)r - cum_q[b];
            q_len = cum_q[b + 1] - cum_q[b];
        } else {
            b = (int)(r / next_n);
            i = (int)(r % next_n);
            q_len = next_n;
        }
        L = seq_lens ? seq_lens[b] : 0;
        vis = dsa_oracle_visible(L, q_len, i);
        kr = k;
        if (topk_lens)
            kr = topk_lens[r] < 0 ? 0 : (topk_lens[r] < k ? topk_lens[r] : k);
        w = wvals ? (window < vis ? window : vis) : 0;
        c = (double*)malloc(sizeof(double) * (size_t)(maxkeys > 0 ? maxkeys : 1) * (size_t)d_qk);
        sc = (double*)malloc(sizeof(double) * (size_t)(maxkeys > 0 ? maxkeys : 1));
        if (!c || !sc) {
            free(c);
            free(sc);
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        for (j = 0; j < kr; ++j) {
            int s = idx[r * idx_stride + j];
            if (s < 0)
                continue;
            if (latent_row(fmt, cvals, vps, vts, cscales, sps, sts, bt, bt_stride, max_pages, page_kv, num_pages,
                           b, s, d_qk, c + (size_t)nkeys * d_qk)) {
#pragma omp atomic write
                err = ORACLE_ERR_PAGE;
                continue;
            }
            ++nkeys;
        }
        for (j = vis - w; j < vis; ++j) {
            if (latent_row(fmt, wvals, wvps, wvts, wscales, wsps, wsts, wbt, wbt_stride, wmax_pages, wpage_kv,
                           wnum_pages, b, j, d_qk, c + (size_t)nkeys * d_qk)) {
#pragma omp atomic write
                err = ORACLE_ERR_PAGE;
                continue;
            }
            ++nkeys;
        }
        for (h = 0; h < Hq; ++h) {
            const uint16_t* qh = q + ((int64_t)r * Hq + h) * d_qk;
            double* o = out + ((int64_t)r * Hq + h) * d_v;
            double m = -INFINITY, l = 0.0, LSE;
            for (d = 0; d < d_v; ++d)
                o[d] = 0.0;
            if (nkeys == 0) {
                lse[(int64_t)r * Hq + h] = -INFINITY;
                continue;
            }
            for (j = 0; j < nkeys; ++j) {
                double dot = 0.0;
                for (d = 0; d < d_qk; ++d)
                    dot += dsa_oracle_bf16(qh[d]) * c[(size_t)j * d_qk + d];
                sc[j] = softmax_scale * dot;
                if (sc[j] > m)
                    m = sc[j];
            }
            for (j = 0; j < nkeys; ++j)
                l += exp(sc[j] - m);
            LSE = m + log(l);
            lse[(int64_t)r * Hq + h] = LSE;
            for (j = 0; j < nkeys; ++j) {
                double pj = exp(sc[j] - LSE);
                for (d = 0; d < d_v; ++d)
                    o[d] += pj * c[(size_t)j * d_qk + d];
            }
        }
        free(c);
        free(sc);
    }
    return err;
}

/* --------------------------------------------- K-cache quantise / scatter */

/* Round-half-to-even of a non-negative double to an integer (the doubles met
 * here are exact multiples of 2^-k with small magnitude, so this is exact). */
static double round_half_even(double a)
{
    double f = floor(a), d = a - f;
    if (d > 0.5)
        return f + 1.0;
    if (d < 0.5)
        return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* Nearest OCP E4M3 ("fn") code to the float v, ties to the even code,
 * saturating to +-448 (no NaN produced for finite v); the sign bit is v's sign
 * bit (so a negative value that rounds to zero gives 0x80).  Each step follows
 * the format: subnormals are multiples of 2^-9 below 2^-6; a normal binade
 * [2^E, 2^(E+1)) holds 8 values spaced 2^(E-3). */
uint8_t dsa_oracle_encode_e4m3(float v)
{
    uint32_t u;
    double a;
    uint8_t sign, code;
    memcpy(&u, &v, sizeof u);
    sign = (uint8_t)((u >> 31) << 7);
    a = fabs((double)v);
    if (a >= 448.0) {
        code = 0x7E;
    } else if (a < ldexp(1.0, -6)) {
        double m = round_half_even(a / ldexp(1.0, -9));        /* 0 .. 8 */
        code = (uint8_t)m;                                     /* m = 8 is 2^-6: code 0x08 */
    } else {
        int E;
        double q;
        frexp(a, &E);                                          /* a = f * 2^E, f in [0.5, 1) */
        E -= 1;                                                /* a in [2^E, 2^(E+1)) */
        q = round_half_even(a / ldexp(1.0, E - 3));            /* 8 .. 16 */
        if (q >= 16.0) {
            q = 8.0;
            E += 1;
        }
        if (E > 8 || (E == 8 && q > 14.0))
            code = 0x7E;                                       /* beyond 448: saturate */
        else
            code = (uint8_t)(((E + 7) << 3) | ((int)q - 8));
    }
    return (uint8_t)(sign | code);
}

/* Nearest OCP E2M1 code (4 bits) to the float v, ties to the even code,
 * saturating to +-6; the sign bit (bit 3) is v's sign bit.  Grid: 0, 0.5, 1,
 * 1.5 (spacing 0.5), 2, 3 (spacing 1), 4, 6 (spacing 2). */
uint8_t dsa_oracle_encode_e2m1(float v)
{
    uint32_t u;
    double a;
    uint8_t sign, code;
    memcpy(&u, &v, sizeof u);
    sign = (uint8_t)((u >> 31) << 3);
    a = fabs((double)v);
    if (a >= 6.0)
        code = 7;
    else if (a < 2.0)
        code = (uint8_t)round_half_even(a * 2.0);              /* 0 .. 4 (4 = 2.0) */
    else if (a < 4.0)
        code = (uint8_t)(round_half_even(a) + 2.0);            /* 2, 3, 4 -> codes 4, 5, 6 */
    else
        code = (uint8_t)(round_half_even(a / 2.0) + 4.0);      /* 2, 3 -> codes 6, 7 */
    return (uint8_t)(sign | code);
}

/* Writes new K rows into a paged cache through a slot mapping (slot = physical
 * page * page_kv + row; slots < 0 are skipped), quantising each row:
 *  - FP8 (fmt 0): per token, amax = max_d |x_d| (fp32), scale = amax / 448 in
 *    fp32 (1 when amax = 0), code_d = e4m3(x_d / scale) with the division in
 *    fp32; the fp32 scale is stored beside the token.
 *  - MXFP4 (fmt 1): per 32-element block, amax (fp32), shared exponent
 *    e = floor(log2 amax) - 2 clamped to [-127, 127] (-127 when amax = 0),
 *    stored as the ue8m0 byte e + 127; element codes e2m1(x_d * 2^-e), packed
 *    two per byte with the even element in the low nibble.
 * k:  [n_tokens] rows of D values, fp32 (k_is_bf16 = 0) or bf16 bits, row
 *     stride k_stride ELEMENTS.  Returns ORACLE_ERR_PAGE if a slot's page is
 *     outside [0, num_pages) (that token is skipped). */
int dsa_oracle_quantize_scatter(const void* k, int k_is_bf16, int64_t k_stride, int n_tokens, int D,
                                const int64_t* slots, int fmt, uint8_t* vals, int64_t vps, int64_t vts,
                                uint8_t* scales, int64_t sps, int64_t sts, int page_kv, int num_pages)
{
    int err = ORACLE_OK;
    long t;
    if (n_tokens < 0 || D <= 0 || page_kv <= 0 || (fmt != 0 && fmt != 1) || (fmt == 1 && D % 32 != 0))
        return ORACLE_ERR_ARG;
    for (t = 0; t < n_tokens; ++t) {
        int64_t slot = slots[t], page, row;
        float x[4096];
        uint8_t *vrow, *srow;
        int d;
        if (slot < 0)
            continue;
        page = slot / page_kv;
        row = slot % page_kv;
        if (page >= num_pages || D > 4096) {
            err = ORACLE_ERR_PAGE;
            continue;
        }
        for (d = 0; d < D; ++d) {
            if (k_is_bf16) {
                uint16_t bits = ((const uint16_t*)k)[t * k_stride + d];
                x[d] = (float)dsa_oracle_bf16(bits);
            } else {
                x[d] = ((const float*)k)[t * k_stride + d];
            }
        }
        vrow = vals + page * vps + row * vts;
        srow = scales + page * sps + row * sts;
        if (fmt == 0) {
            float amax = 0.0f, scale;
            for (d = 0; d < D; ++d)
                if (fabsf(x[d]) > amax)
                    amax = fabsf(x[d]);
            scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            for (d = 0; d < D; ++d) {
                float q = x[d] / scale;
                vrow[d] = dsa_oracle_encode_e4m3(q);
            }
            memcpy(srow, &scale, sizeof scale);
        } else {
            int blk;
            for (blk = 0; blk < D / 32; ++blk) {
                float amax = 0.0f;
                int e;
                for (d = 32 * blk; d < 32 * blk + 32; ++d)
                    if (fabsf(x[d]) > amax)
                        amax = fabsf(x[d]);
                if (amax > 0.0f) {
                    int E;
                    frexpf(amax, &E);                  /* amax = f * 2^E, f in [0.5, 1) */
                    e = (E - 1) - 2;
                } else {
                    e = -127;
                }
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
                srow[blk] = (uint8_t)(e + 127);
                for (d = 32 * blk; d < 32 * blk + 32; d += 2) {
                    uint8_t lo = dsa_oracle_encode_e2m1((float)ldexp((double)x[d], -e));
                    uint8_t hi = dsa_oracle_encode_e2m1((float)ldexp((double)x[d + 1], -e));
                    vrow[d / 2] = (uint8_t)(lo | (hi << 4));
                }
            }
        }
    }
    return err;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int dsa_oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
