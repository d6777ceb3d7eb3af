// noalloc.cu -- indexer logits for callers that cannot allocate device memory.
//
// indexer_mqa_logits_paged() needs a caller-owned schedule buffer (built by
// dsa_indexer_build_schedule()) for calls of more than 256 work units.  Some
// callers cannot provide one: code that runs inside a framework whose allocator
// owns all device memory and offers no hook for a plugin, or an inference host
// that must not call cudaMalloc on its request path.  This file keeps the
// schedule in a fixed, file-scope device array instead and runs the same two
// launches (schedule build, then logits) on it.
//
// The array is part of the library's device code: it comes into being on a GPU
// when the library's module is loaded there, which is at the latest on the
// first call of this entry point with that GPU current, and it stays until the
// process exits.  Host code cannot use the symbol's name as a device address,
// so the address is looked up with cudaGetSymbolAddress at set-up: once per
// device and CUDA context, on the first call made while that device is current
// (again after a device reset, which creates a new context).  That first call
// must therefore come before any stream capture.
#include <cuda.h>
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
struct ScratchSlot {
    unsigned long long ctx_id;   // CUDA context the address belongs to (0 = not set up)
    void* ptr;
};
ScratchSlot g_slot[kMaxDev] = {};
std::mutex g_sched_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if it cannot be
// read); a device reset replaces the context and so changes the id.
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_sched_scratch on the current device.  Set up once per
// device and context: cudaGetSymbolAddress with that device current (it loads
// the module there if needed and allocates nothing), its return code checked.
dsa_status scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDev)
        return DSA_ERR_UNSUPPORTED;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_sched_mu);
    ScratchSlot& slot = g_slot[dev];
    if (!slot.ptr || ctx == 0 || slot.ctx_id != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_sched_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e);
        slot.ptr = ptr;
        // the lookup made the device's context current if it was not yet
        slot.ctx_id = current_context_id();
    }
    *out = slot.ptr;
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
    // every check of the regular entry point first: a rejected call enqueues
    // nothing and leaves the fixed array as it was
    int64_t units = 0;
    dsa_status st = validate_logits_call(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                         row_begin, row_end, logits, logits_row_stride, logits_width, &units);
    if (st != DSA_OK)
        return st;
    if (sched_bytes_for_units(units) > static_cast<int64_t>(kNoallocSchedBytes))
        return DSA_ERR_CAPACITY;             // too many work units for the fixed array
    // small calls: the logits kernel builds its units itself (one launch, the array untouched)
    if (units <= kInlineUnits)
        return indexer_mqa_logits_paged(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                        row_begin, row_end, nullptr, 0, logits, logits_row_stride, logits_width,
                                        status_dev, stream);
    void* sched = nullptr;
    st = scratch_address(&sched);
    if (st != DSA_OK)
        return st;
    // every word the logits kernel reads is rewritten by the schedule build first,
    // so nothing has to be cleared between calls
    st = dsa_indexer_build_schedule(context_lens, batch, next_n, num_heads, k->compress_ratio, row_begin, row_end,
                                    sched, kNoallocSchedBytes, status_dev, stream);
    if (st != DSA_OK)
        return st;
    return indexer_mqa_logits_paged(q, q_scales, q_fmt, weights, num_heads, k, context_lens, batch, next_n,
                                    row_begin, row_end, sched, kNoallocSchedBytes, logits, logits_row_stride,
                                    logits_width, status_dev, stream);
}
