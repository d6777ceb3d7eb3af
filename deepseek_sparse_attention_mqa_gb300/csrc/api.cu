// api.cu -- the extern "C" entry points of libdsa: host-side validation (no
// device synchronisation, nothing enqueued on error), device queries, tensor-map
// encoding and dispatch to the kernel launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/dsa.h"
#include "common.cuh"
#include "host.h"

namespace dsa {

static thread_local int g_last_cuda_error = 0;

dsa_status cuda_fail(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return DSA_ERR_CUDA;
}

dsa_status check_launch()
{
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

namespace {

constexpr int kMaxDevices = 64;
struct DevSlot {
    std::atomic<int> ready{0};
    DeviceInfo info;
};
DevSlot g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxRatio = 65536;

// Tokens per entry of an indexer K cache: its compress_ratio, 0 and 1 both
// meaning one entry per token; -1 if out of range.
int ratio_of(int32_t r)
{
    if (r < 0 || r > kMaxRatio)
        return -1;
    return r <= 1 ? 1 : r;
}

}  // namespace

dsa_status current_device(DeviceInfo* out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices)
        return DSA_ERR_UNSUPPORTED;
    DevSlot& slot = g_dev[dev];
    if (!slot.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!slot.ready.load(std::memory_order_relaxed)) {
            DeviceInfo d;
            d.ordinal = dev;
            if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                    cudaSuccess)
                return cuda_fail(e);
            slot.info = d;
            slot.ready.store(1, std::memory_order_release);
        }
    }
    *out = slot.info;
    // the kernels are built for sm_103a only
    if (out->cc_major != 10 || out->cc_minor != 3)
        return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

dsa_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return DSA_ERR_UNSUPPORTED;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank)
            gs[i] = strides_bytes[i];
    }
    const CUresult r = fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_INVALID_ARG;
}

// ---------------------------------------------------------------- validation

static bool heads_supported(int h)
{
    return h == 4 || h == 8 || h == 16 || h == 32 || h == 64 || h == 128;
}

static bool row_range_ok(int batch, int next_n, int row_begin, int row_end)
{
    if (batch < 0 || next_n < 1 || row_begin < 0 || row_end < row_begin)
        return false;
    return static_cast<int64_t>(row_end) <= static_cast<int64_t>(batch) * next_n &&
           static_cast<int64_t>(batch) * next_n < (int64_t(1) << 31);
}

// Paged-cache checks shared by the indexer and MLA paths.  The indexer copies
// whole pages with TMA (page_kv 32 or 64); the MLA gathers token by token and
// takes any page size (e.g. a compressed cache holding a few entries per
// physical block).
static dsa_status check_cache(const dsa_paged_cache* c, bool need_scales, bool any_page = false)
{
    if (!c || !c->values || !c->block_table)
        return DSA_ERR_INVALID_ARG;
    if (any_page ? c->page_kv < 1 : (c->page_kv != 32 && c->page_kv != 64))
        return DSA_ERR_UNSUPPORTED;
    if (c->num_pages < 1 || c->head_dim < 1 || c->max_pages_per_seq < 1 ||
        c->bt_row_stride < c->max_pages_per_seq)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(c->values) || c->val_page_stride % 16 != 0 || c->val_page_stride <= 0)
        return DSA_ERR_INVALID_ARG;
    // the indexer copies token scales 16 bytes at a time; the MLA reads one fp32 per token
    const int64_t sc_align = any_page ? 4 : 16;
    if (need_scales && (!c->scales || (reinterpret_cast<uintptr_t>(c->scales) % sc_align) != 0 ||
                        c->sc_page_stride % sc_align != 0 || c->sc_page_stride <= 0))
        return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

// Every host-side check of a logits call except those on the schedule buffer:
// the same for indexer_mqa_logits_paged and its allocation-free variant, so
// that both reject a bad call before enqueueing anything.  On success *units is
// the call's work-unit count.
dsa_status validate_logits_call(const void* q, const void* q_scales, int q_fmt, const float* weights,
                                int num_heads, const dsa_paged_cache* k, const int32_t* context_lens, int batch,
                                int next_n, int row_begin, int row_end, const float* logits,
                                int64_t logits_row_stride, int logits_width, int64_t* units)
{
    if (!row_range_ok(batch, next_n, row_begin, row_end) || !k)
        return DSA_ERR_INVALID_ARG;
    if (!heads_supported(num_heads))
        return DSA_ERR_UNSUPPORTED;
    if (q_fmt != k->fmt || (q_fmt != DSA_KV_FP8_E4M3 && q_fmt != DSA_KV_MXFP4))
        return DSA_ERR_UNSUPPORTED;
    const int D = k->head_dim;
    if (D != 32 && D != 64 && D != 128)
        return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_cache(k, true);
    if (st != DSA_OK)
        return st;
    if (ratio_of(k->compress_ratio) < 0)
        return DSA_ERR_INVALID_ARG;
    if (q_fmt == DSA_KV_FP8_E4M3) {
        if (k->val_token_stride != D || k->sc_token_stride != 4 || k->val_page_stride < int64_t(k->page_kv) * D ||
            k->sc_page_stride < int64_t(k->page_kv) * 4)
            return DSA_ERR_INVALID_ARG;
    } else {
        if (k->val_token_stride != D / 2 || k->sc_token_stride != D / 32 ||
            k->val_page_stride < int64_t(k->page_kv) * (D / 2) || k->sc_page_stride < int64_t(k->page_kv) * (D / 32) ||
            !q_scales)
            return DSA_ERR_INVALID_ARG;
    }
    // MXFP4 keeps one TMEM accumulator per 32-element block: head_dim 128 fits
    // units of at most 128 columns (rows x heads) in the 512 TMEM columns
    if (q_fmt == DSA_KV_MXFP4 && D == 128 && unit_rows(next_n, num_heads) * num_heads > 128)
        return DSA_ERR_UNSUPPORTED;
    if (!q || !aligned16(q) || !weights || !aligned16(weights) || !logits || (batch > 0 && !context_lens))
        return DSA_ERR_INVALID_ARG;
    if (logits_width < 0 || logits_row_stride < logits_width)
        return DSA_ERR_INVALID_ARG;
    *units = count_units(batch, next_n, unit_rows(next_n, num_heads), row_begin, row_end);
    return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(dsa_status s)
{
    switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CAPACITY: return "DSA_ERR_CAPACITY";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    }
    return "DSA_ERR_UNKNOWN";
}

int dsa_last_cuda_error(void) { return g_last_cuda_error; }

int dsa_version(void) { return 200; }

size_t dsa_indexer_schedule_bytes(int batch, int next_n, int num_heads, int row_begin, int row_end)
{
    if (!row_range_ok(batch, next_n, row_begin, row_end) || num_heads < 1 || num_heads > kMaxUnitCols)
        return 0;
    const int G = unit_rows(next_n, num_heads);
    return static_cast<size_t>(sched_bytes_for_units(count_units(batch, next_n, G, row_begin, row_end)));
}

dsa_status dsa_indexer_build_schedule(const int32_t* context_lens, int batch, int next_n, int num_heads,
                                      int compress_ratio, int row_begin, int row_end, void* sched,
                                      size_t sched_bytes, int32_t* status_dev, void* stream)
{
    if (!row_range_ok(batch, next_n, row_begin, row_end) || num_heads < 1 || num_heads > kMaxUnitCols)
        return DSA_ERR_INVALID_ARG;
    const int ratio = ratio_of(compress_ratio);
    if (ratio < 0)
        return DSA_ERR_INVALID_ARG;
    if (!sched || !aligned16(sched) || (batch > 0 && !context_lens))
        return DSA_ERR_INVALID_ARG;
    const int G = unit_rows(next_n, num_heads);
    const int64_t units = count_units(batch, next_n, G, row_begin, row_end);
    if (units > (int64_t(1) << 30))
        return DSA_ERR_UNSUPPORTED;
    if (sched_bytes < static_cast<size_t>(sched_bytes_for_units(units)))
        return DSA_ERR_CAPACITY;
    DeviceInfo dev;
    dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    return launch_build_schedule(context_lens, batch, next_n, ratio, G, row_begin, row_end, static_cast<int>(units),
                                 static_cast<int32_t*>(sched), status_dev, static_cast<cudaStream_t>(stream));
}

// The logits launch shared by indexer_mqa_logits_paged and indexer_score_topk
// (topk.k = 0: logits only); the call has passed validate_logits_call.
static dsa_status launch_logits_call(const void* q, const void* q_scales, int q_fmt, const float* weights,
                                     int num_heads, const dsa_paged_cache* k, const int32_t* context_lens, int batch,
                                     int next_n, int row_begin, int row_end, int64_t units, const void* sched,
                                     float* logits, int64_t logits_row_stride, int logits_width,
                                     const FusedTopk& topk, int32_t* status_dev, void* stream)
{
    DeviceInfo dev;
    const dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    LogitsArgs a;
    a.q = q;
    a.q_scales = q_scales;
    a.weights = weights;
    a.num_heads = num_heads;
    a.k = k;
    a.context_lens = context_lens;
    a.batch = batch;
    a.next_n = next_n;
    a.row_begin = row_begin;
    a.row_end = row_end;
    a.rows_per_unit = unit_rows(next_n, num_heads);
    a.num_units = static_cast<int>(units);
    a.ratio = ratio_of(k->compress_ratio);
    a.sched = static_cast<const int32_t*>(sched);
    a.logits = logits;
    a.logits_row_stride = logits_row_stride;
    a.logits_width = logits_width;
    a.status = status_dev;
    a.topk = topk;
    if (q_fmt == DSA_KV_FP8_E4M3)
        return launch_logits_fp8(a, dev, static_cast<cudaStream_t>(stream));
    return launch_logits_mxfp4(a, dev, static_cast<cudaStream_t>(stream));
}

dsa_status indexer_mqa_logits_paged(const void* q, const void* q_scales, int q_fmt, const float* weights,
                                    int num_heads, const dsa_paged_cache* k, const int32_t* context_lens,
                                    int batch, int next_n, int row_begin, int row_end, const void* sched,
                                    size_t sched_bytes, float* logits, int64_t logits_row_stride,
                                    int logits_width, int32_t* status_dev, void* stream)
{
    int64_t units = 0;
    dsa_status st = validate_logits_call(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                         row_begin, row_end, logits, logits_row_stride, logits_width, &units);
    if (st != DSA_OK)
        return st;
    if (sched && !aligned16(sched))
        return DSA_ERR_INVALID_ARG;
    if (sched && sched_bytes < static_cast<size_t>(sched_bytes_for_units(units)))
        return DSA_ERR_CAPACITY;
    if (!sched && units > kInlineUnits)      // the kernels build at most kInlineUnits units themselves
        return DSA_ERR_CAPACITY;
    if (row_end == row_begin)
        return DSA_OK;
    const FusedTopk none{0, nullptr, 0, nullptr, nullptr};
    return launch_logits_call(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n, row_begin,
                              row_end, units, sched, logits, logits_row_stride, logits_width, none, status_dev,
                              stream);
}

size_t dsa_score_topk_workspace_bytes(int batch, int next_n, int num_heads, int row_begin, int row_end)
{
    if (!row_range_ok(batch, next_n, row_begin, row_end) || num_heads < 1 || num_heads > kMaxUnitCols)
        return 0;
    const int64_t units = count_units(batch, next_n, unit_rows(next_n, num_heads), row_begin, row_end);
    return static_cast<size_t>((units * 4 + 15) / 16 * 16 + 16);
}

dsa_status indexer_score_topk(const void* q, const void* q_scales, int q_fmt, const float* weights, int num_heads,
                              const dsa_paged_cache* k, const int32_t* context_lens, int batch, int next_n,
                              int row_begin, int row_end, const void* sched, size_t sched_bytes, float* logits,
                              int64_t logits_row_stride, int logits_width, int topk, int32_t* idx,
                              int64_t idx_row_stride, int32_t* count, void* workspace, size_t ws_bytes,
                              int32_t* status_dev, void* stream)
{
    int64_t units = 0;
    dsa_status st = validate_logits_call(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                         row_begin, row_end, logits, logits_row_stride, logits_width, &units);
    if (st != DSA_OK)
        return st;
    if (topk < 1 || topk > 16384)
        return DSA_ERR_UNSUPPORTED;
    if (!idx || idx_row_stride < topk || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
        return DSA_ERR_INVALID_ARG;
    // the selection streams logits rows with 16-byte loads
    if (!aligned16(logits) || logits_row_stride % 4 != 0)
        return DSA_ERR_INVALID_ARG;
    if (sched && !aligned16(sched))
        return DSA_ERR_INVALID_ARG;
    if (sched && sched_bytes < static_cast<size_t>(sched_bytes_for_units(units)))
        return DSA_ERR_CAPACITY;
    if (!sched && units > kInlineUnits)
        return DSA_ERR_CAPACITY;
    if (ws_bytes < dsa_score_topk_workspace_bytes(batch, next_n, num_heads, row_begin, row_end))
        return DSA_ERR_CAPACITY;
    if (row_end == row_begin)
        return DSA_OK;
    const FusedTopk f{topk, idx, idx_row_stride, count, static_cast<int32_t*>(workspace)};
    return launch_logits_call(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n, row_begin,
                              row_end, units, sched, logits, logits_row_stride, logits_width, f, status_dev, stream);
}

size_t dsa_topk_workspace_bytes(int rows, int logits_width, int k)
{
    (void)rows;
    (void)logits_width;
    (void)k;
    return 0;
}

dsa_status indexer_topk(const float* logits, int64_t logits_row_stride, int logits_width,
                        const int32_t* context_lens, int batch, int next_n, int compress_ratio, int row_begin,
                        int row_end, int k, int32_t* idx, int64_t idx_row_stride, int32_t* count, void* workspace,
                        size_t ws_bytes, int32_t* status_dev, void* stream)
{
    (void)workspace;
    (void)ws_bytes;
    if (!row_range_ok(batch, next_n, row_begin, row_end))
        return DSA_ERR_INVALID_ARG;
    const int ratio = ratio_of(compress_ratio);
    if (ratio < 0)
        return DSA_ERR_INVALID_ARG;
    if (k < 1 || k > 16384)
        return DSA_ERR_UNSUPPORTED;
    if (!logits || !idx || logits_width < 0 || logits_row_stride < logits_width || idx_row_stride < k ||
        (batch > 0 && !context_lens))
        return DSA_ERR_INVALID_ARG;
    if (row_end == row_begin)
        return DSA_OK;
    DeviceInfo dev;
    dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    TopkArgs a;
    a.logits = logits;
    a.logits_row_stride = logits_row_stride;
    a.logits_width = logits_width;
    a.context_lens = context_lens;
    a.batch = batch;
    a.next_n = next_n;
    a.row_begin = row_begin;
    a.row_end = row_end;
    a.ratio = ratio;
    a.k = k;
    a.idx = idx;
    a.idx_row_stride = idx_row_stride;
    a.count = count;
    a.status = status_dev;
    return launch_topk(a, dev, static_cast<cudaStream_t>(stream));
}

size_t dsa_sparse_mla_workspace_bytes(int rows, int num_heads, int d_qk, int d_v, int k)
{
    (void)rows;
    (void)num_heads;
    (void)d_qk;
    (void)d_v;
    (void)k;
    return 0;
}

// Host checks of one MLA latent cache (fmt FP8 + token scale, or bf16).
static dsa_status check_mla_cache(const dsa_paged_cache* kv, int d_qk)
{
    if (!kv)
        return DSA_ERR_INVALID_ARG;
    if (kv->fmt != DSA_KV_FP8_E4M3 && kv->fmt != DSA_KV_BF16)
        return DSA_ERR_UNSUPPORTED;
    if (kv->head_dim != d_qk)
        return DSA_ERR_INVALID_ARG;
    const bool fp8 = kv->fmt == DSA_KV_FP8_E4M3;
    dsa_status st = check_cache(kv, fp8, true);
    if (st != DSA_OK)
        return st;
    const int64_t row_bytes = fp8 ? d_qk : 2 * int64_t(d_qk);
    if (kv->val_token_stride < row_bytes || kv->val_page_stride < kv->page_kv * kv->val_token_stride)
        return DSA_ERR_INVALID_ARG;
    if (fp8 && (kv->sc_token_stride < 4 || kv->sc_token_stride % 4 != 0))
        return DSA_ERR_INVALID_ARG;
    // positions and indices are tagged with bit 30 inside the kernels
    if (static_cast<int64_t>(kv->max_pages_per_seq) * kv->page_kv >= (int64_t(1) << 30))
        return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

static dsa_status run_sparse_mla(MlaArgs& a, void* stream)
{
    if (a.rows == 0)
        return DSA_OK;
    DeviceInfo dev;
    const dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    const bool tc_layout = aligned16(a.q) && aligned16(a.out) && a.kv->val_token_stride % 16 == 0 &&
                           (!a.swa || a.swa->val_token_stride % 16 == 0);
    if (sparse_mla_tc_supported(a) && tc_layout)
        return launch_sparse_mla_tc(a, dev, static_cast<cudaStream_t>(stream));
    return launch_sparse_mla_simt(a, static_cast<cudaStream_t>(stream));
}

dsa_status sparse_mla_decode(const void* q_bf16, int rows, int num_heads, int d_qk, int d_v, float softmax_scale,
                             const dsa_paged_cache* kv, const int32_t* seq_of_row, int next_n, const int32_t* idx,
                             int64_t idx_row_stride, int k, void* out_bf16, float* lse, void* workspace,
                             size_t ws_bytes, int32_t* status_dev, void* stream)
{
    if (rows < 0 || num_heads < 1 || k < 0 || !kv || (!seq_of_row && next_n < 1))
        return DSA_ERR_INVALID_ARG;
    if (d_qk < 16 || d_qk > 1024 || d_qk % 16 != 0 || d_v < 16 || d_v % 16 != 0 || d_v > d_qk || d_v > 512)
        return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_mla_cache(kv, d_qk);
    if (st != DSA_OK)
        return st;
    if (rows > 0 && (!q_bf16 || !idx || !out_bf16 || !lse || idx_row_stride < k))
        return DSA_ERR_INVALID_ARG;
    if (ws_bytes < dsa_sparse_mla_workspace_bytes(rows, num_heads, d_qk, d_v, k))
        return DSA_ERR_CAPACITY;
    MlaArgs a{};
    a.q = q_bf16;
    a.rows = rows;
    a.num_heads = num_heads;
    a.d_qk = d_qk;
    a.d_v = d_v;
    a.softmax_scale = softmax_scale;
    a.kv = kv;
    a.seq_of_row = seq_of_row;
    a.next_n = next_n;
    a.idx = idx;
    a.idx_row_stride = idx_row_stride;
    a.k = k;
    a.out = out_bf16;
    a.lse = lse;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.status = status_dev;
    return run_sparse_mla(a, stream);
}

dsa_status sparse_mla_decode_swa(const void* q_bf16, int rows, int num_heads, int d_qk, int d_v, float softmax_scale,
                                 const dsa_paged_cache* kv, const int32_t* idx, int64_t idx_row_stride, int k,
                                 const int32_t* topk_lens, const dsa_paged_cache* swa, int window,
                                 const int32_t* seq_lens, const int32_t* cum_seq_lens_q, int batch, int next_n,
                                 void* out_bf16, float* lse, void* workspace, size_t ws_bytes, int32_t* status_dev,
                                 void* stream)
{
    if (rows < 0 || num_heads < 1 || k < 0 || !kv || batch < 0 || (!cum_seq_lens_q && next_n < 1))
        return DSA_ERR_INVALID_ARG;
    if (d_qk < 16 || d_qk > 1024 || d_qk % 16 != 0 || d_v < 16 || d_v % 16 != 0 || d_v > d_qk || d_v > 512)
        return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_mla_cache(kv, d_qk);
    if (st != DSA_OK)
        return st;
    if (swa) {
        st = check_mla_cache(swa, d_qk);
        if (st != DSA_OK)
            return st;
        if (swa->fmt != kv->fmt)
            return DSA_ERR_UNSUPPORTED;
        if (window < 1 || !seq_lens)
            return DSA_ERR_INVALID_ARG;
    }
    if (!cum_seq_lens_q && static_cast<int64_t>(rows) > static_cast<int64_t>(batch) * next_n)
        return DSA_ERR_INVALID_ARG;
    if (rows > 0 && (!q_bf16 || (k > 0 && !idx) || !out_bf16 || !lse || (k > 0 && idx_row_stride < k)))
        return DSA_ERR_INVALID_ARG;
    if (ws_bytes < dsa_sparse_mla_workspace_bytes(rows, num_heads, d_qk, d_v, k))
        return DSA_ERR_CAPACITY;
    MlaArgs a{};
    a.q = q_bf16;
    a.rows = rows;
    a.num_heads = num_heads;
    a.d_qk = d_qk;
    a.d_v = d_v;
    a.softmax_scale = softmax_scale;
    a.kv = kv;
    a.seq_of_row = nullptr;
    a.next_n = next_n;
    a.idx = idx;
    a.idx_row_stride = idx_row_stride;
    a.k = k;
    a.out = out_bf16;
    a.lse = lse;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.status = status_dev;
    a.topk_lens = topk_lens;
    a.swa = swa;
    a.window = swa ? window : 0;
    a.seq_lens = seq_lens;
    a.cum_q = cum_seq_lens_q;
    a.batch = batch;
    return run_sparse_mla(a, stream);
}

dsa_status dsa_kv_quantize_scatter(const void* k_new, int k_dtype, int64_t k_row_stride, int n_tokens,
                                   const int64_t* slot_mapping, const dsa_paged_cache* cache, int32_t* status_dev,
                                   void* stream)
{
    if (!cache || n_tokens < 0 || (k_dtype != DSA_DTYPE_F32 && k_dtype != DSA_DTYPE_BF16))
        return DSA_ERR_INVALID_ARG;
    const int D = cache->head_dim;
    const int64_t esize = k_dtype == DSA_DTYPE_BF16 ? 2 : 4;
    if (cache->fmt == DSA_KV_FP8_E4M3) {
        if (D < 8 || D % 8 != 0 || D > 4096)
            return DSA_ERR_UNSUPPORTED;
        if (cache->val_token_stride < D || cache->val_token_stride % 8 != 0 || cache->val_page_stride % 8 != 0 ||
            cache->sc_token_stride < 4 || cache->sc_token_stride % 4 != 0 || cache->sc_page_stride % 4 != 0)
            return DSA_ERR_INVALID_ARG;
    } else if (cache->fmt == DSA_KV_MXFP4) {
        if (D < 32 || D % 32 != 0 || D > 4096)
            return DSA_ERR_UNSUPPORTED;
        if (cache->val_token_stride < D / 2 || cache->val_token_stride % 4 != 0 || cache->val_page_stride % 4 != 0 ||
            cache->sc_token_stride < D / 32)
            return DSA_ERR_INVALID_ARG;
    } else {
        return DSA_ERR_UNSUPPORTED;
    }
    if (cache->page_kv < 1 || cache->num_pages < 1 || !cache->values || !cache->scales ||
        (reinterpret_cast<uintptr_t>(cache->values) & 7u) != 0 ||
        (reinterpret_cast<uintptr_t>(cache->scales) & 3u) != 0 ||
        static_cast<int64_t>(cache->page_kv) * cache->val_token_stride > cache->val_page_stride ||
        static_cast<int64_t>(cache->page_kv) * cache->sc_token_stride > cache->sc_page_stride)
        return DSA_ERR_INVALID_ARG;
    if (n_tokens == 0)
        return DSA_OK;
    if (!k_new || !slot_mapping || !aligned16(k_new) || k_row_stride < D || (k_row_stride * esize) % 16 != 0)
        return DSA_ERR_INVALID_ARG;
    DeviceInfo dev;
    const dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    return launch_kv_scatter(k_new, k_dtype == DSA_DTYPE_BF16, k_row_stride, n_tokens, slot_mapping, cache,
                             status_dev, static_cast<cudaStream_t>(stream));
}

dsa_status dsa_get_device_status(const int32_t* status_dev, int32_t* host_out, void* stream)
{
    if (!status_dev || !host_out)
        return DSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return cuda_fail(e);
    e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // extern "C"
