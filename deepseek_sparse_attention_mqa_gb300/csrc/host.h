// host.h -- internal host-side helpers shared by the launchers (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dsa.h"
#include "common.cuh"

namespace dsa {

// Record a CUDA error for dsa_last_cuda_error() and map it to DSA_ERR_CUDA.
dsa_status cuda_fail(cudaError_t e);
// Check the last launch on this thread.
dsa_status check_launch();

// Properties of the current device, cached per device ordinal.
struct DeviceInfo {
    int ordinal;
    int sm_count;
    int cc_major;
    int cc_minor;
    int max_smem_optin;
};
dsa_status current_device(DeviceInfo* out);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// dims / box are innermost-first; strides (bytes) are for dims 1..rank-1.
dsa_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle);

// Host checks of a logits call shared by its entry points (api.cu); *units
// receives the call's work-unit count.
dsa_status validate_logits_call(const void* q, const void* q_scales, int q_fmt, const float* weights,
                                int num_heads, const dsa_paged_cache* k, const int32_t* context_lens, int batch,
                                int next_n, int row_begin, int row_end, const float* logits,
                                int64_t logits_row_stride, int logits_width, int64_t* units);

// Launchers implemented in the kernel translation units.
dsa_status launch_build_schedule(const int32_t* context_lens, int batch, int next_n, int ratio,
                                 int rows_per_unit, int row_begin, int row_end, int num_units,
                                 int32_t* sched, int32_t* status, cudaStream_t stream);

struct LogitsArgs {
    const void* q;
    const void* q_scales;
    const float* weights;
    int num_heads;
    const dsa_paged_cache* k;
    const int32_t* context_lens;
    int batch;
    int next_n;
    int row_begin;
    int row_end;
    int rows_per_unit;
    int num_units;
    int ratio;                  // tokens per K-cache entry
    const int32_t* sched;
    float* logits;
    int64_t logits_row_stride;
    int logits_width;
    int32_t* status;
    FusedTopk topk;             // k = 0: logits only
};
dsa_status launch_logits_fp8(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream);
dsa_status launch_logits_mxfp4(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream);

struct TopkArgs {
    const float* logits;
    int64_t logits_row_stride;
    int logits_width;
    const int32_t* context_lens;
    int batch;
    int next_n;
    int row_begin;
    int row_end;
    int ratio;                  // tokens per K-cache entry
    int k;
    int32_t* idx;
    int64_t idx_row_stride;
    int32_t* count;
    int32_t* status;
};
dsa_status launch_topk(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream);

dsa_status launch_kv_scatter(const void* k, bool bf16, int64_t k_stride, int n_tokens, const int64_t* slots,
                             const dsa_paged_cache* c, int32_t* status, cudaStream_t stream);

struct MlaArgs {
    const void* q;
    int rows;
    int num_heads;
    int d_qk;
    int d_v;
    float softmax_scale;
    const dsa_paged_cache* kv;
    const int32_t* seq_of_row;
    int next_n;
    const int32_t* idx;
    int64_t idx_row_stride;
    int k;
    void* out;
    float* lse;
    void* workspace;
    size_t ws_bytes;
    int32_t* status;
    // sliding window and dynamic lengths (all null / 0: plain sparse MLA)
    const int32_t* topk_lens;       // [rows]: leading entries of idx to use
    const dsa_paged_cache* swa;     // window cache
    int window;
    const int32_t* seq_lens;        // [batch]
    const int32_t* cum_q;           // [batch + 1]
    int batch;
};
dsa_status launch_sparse_mla_simt(const MlaArgs& a, cudaStream_t stream);
bool sparse_mla_tc_supported(const MlaArgs& a);
dsa_status launch_sparse_mla_tc(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace dsa
