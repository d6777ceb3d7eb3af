// noalloc.cu -- indexer logits for callers that cannot allocate device memory.
//
// indexer_mqa_logits_paged() needs a caller-owned schedule buffer (built by
// dsa_indexer_build_schedule()).  Some callers cannot provide one: code that
// runs inside a framework whose allocator owns all device memory and offers no
// hook for a plugin, or an inference host that must not call cudaMalloc on its
// request path.  This file keeps the schedule in a fixed, file-scope device array
// instead and runs the same two launches (schedule build, then logits) on it.
//
// The array is allocated when the library is loaded, on every GPU the process
// uses, and stays until the process exits.  Its device address is looked up
// with cudaGetSymbolAddress once per device, on the first call made while that
// device is current.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/dsa.h"
#include "common.cuh"
#include "host.h"

namespace dsa {
namespace {

// 256 KiB: 32 header bytes + 32 bytes per work unit -> up to 8191 units
// (e.g. a decode batch of 8191 sequences, or a prefill chunk of 32764 rows at
// 64 heads).
constexpr size_t kNoallocSchedBytes = 256 * 1024;

static __device__ __align__(256) int32_t g_sched_scratch[kNoallocSchedBytes / 4];

constexpr int kMaxDev = 64;
void* g_sched_ptr[kMaxDev] = {};
std::mutex g_sched_mu;

// Device address of g_sched_scratch on the current device (looked up once per device).
dsa_status scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDev)
        return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_sched_mu);
    if (!g_sched_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_sched_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e);
        g_sched_ptr[dev] = ptr;
    }
    *out = g_sched_ptr[dev];
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" DSA_API dsa_status indexer_mqa_logits_paged_noalloc(
    const void* q, const void* q_scales, int q_fmt, const float* weights, int num_heads,
    const dsa_paged_cache* k, const int32_t* context_lens, int batch, int next_n, int row_begin,
    int row_end, float* logits, int64_t logits_row_stride, int logits_width, int32_t* status_dev,
    void* stream)
{
    const size_t need = dsa_indexer_schedule_bytes(batch, next_n, num_heads, row_begin, row_end);
    if (need == 0)
        return DSA_ERR_INVALID_ARG;
    if (need > kNoallocSchedBytes)
        return DSA_ERR_CAPACITY;             // too many work units for the fixed array
    // small calls: the logits kernel builds its units itself (one launch, the array untouched)
    if (need <= static_cast<size_t>(sched_bytes_for_units(kInlineUnits)))
        return indexer_mqa_logits_paged(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                        row_begin, row_end, nullptr, 0, logits, logits_row_stride, logits_width,
                                        status_dev, stream);
    void* sched = nullptr;
    dsa_status st = scratch_address(&sched);
    if (st != DSA_OK)
        return st;
    // every word the logits kernel reads is rewritten by the schedule build first,
    // so nothing has to be cleared between calls
    st = dsa_indexer_build_schedule(context_lens, batch, next_n, num_heads, row_begin, row_end, sched,
                                    kNoallocSchedBytes, status_dev, stream);
    if (st != DSA_OK)
        return st;
    return indexer_mqa_logits_paged(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                    row_begin, row_end, sched, kNoallocSchedBytes, logits, logits_row_stride,
                                    logits_width, status_dev, stream);
}
