// logits_mxfp4.cu -- paged lightning-indexer MQA logits over an MXFP4 K cache.
#include "common.cuh"
#include "host.h"

namespace dsa {

dsa_status launch_logits_mxfp4(const LogitsArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    (void)a;
    (void)dev;
    (void)stream;
    return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
