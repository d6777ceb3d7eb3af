// selftest.cu -- a check of the bounded on-chip waits every kernel relies on.
//
// Every wait in libdsa's kernels (on an mbarrier fed by copies, MMAs or other
// warps) gives up after a time limit, reports DSA_DEV_TIMEOUT in the caller's
// status word and lets the kernel wind down, so that a lost arrival never hangs
// the GPU.  This kernel runs the same wait helper on a condition the host
// controls: its mbarrier is arrived on only if a device word holds the expected
// value, so a caller that never sets that word sees the wait run out, the
// status bit set and the kernel return -- with the context still usable.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"
#include "ptx.cuh"

namespace dsa {
namespace {

__global__ void wait_selftest_kernel(const int32_t* __restrict__ flag, int32_t expect, uint64_t limit_ns,
                                     int32_t* __restrict__ status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x != 0)
        return;
    // the one arrival the barrier expects happens only under the host's condition
    const int32_t v = *reinterpret_cast<const volatile int32_t*>(flag);
    if (v == expect)
        mbar_arrive(smem_u32(&bar));
    if (!mbar_wait_for(smem_u32(&bar), 0, limit_ns) && status)
        atomicOr(status, DSA_DEV_TIMEOUT);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" DSA_API dsa_status dsa_wait_selftest(const int32_t* flag, int32_t expect, int limit_us,
                                                int32_t* status_dev, void* stream)
{
    if (!flag || !status_dev || limit_us < 1 || static_cast<uint64_t>(limit_us) * 1000ull > kWaitLimitNs)
        return DSA_ERR_INVALID_ARG;
    DeviceInfo dev;
    const dsa_status st = current_device(&dev);
    if (st != DSA_OK)
        return st;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        flag, expect, static_cast<uint64_t>(limit_us) * 1000ull, status_dev);
    return check_launch();
}
