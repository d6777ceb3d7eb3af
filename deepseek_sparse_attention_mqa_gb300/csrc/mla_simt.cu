// mla_simt.cu -- sparse MLA decode on CUDA cores, for head counts / head dims the
// tensor-core kernel does not cover (small heads, d_qk not a multiple of 64).
//
// "Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels" (flashinfer #3269): attention
// of each query row over its top-k selected latent tokens, natural-log LSE,
// bf16 output; an index < 0 marks an unused slot.
//
// One CTA per (row, group of 16 heads), 8 warps with 2 heads each.  Selected
// latent rows are gathered 32 at a time through the block table, decoded to
// fp32 (e4m3 * token scale, or bf16) into shared memory, and every warp runs an
// online softmax over them for its heads with the head dimension split across
// lanes.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerCta = 16;
constexpr int kHeadsPerWarp = kHeadsPerCta / (kThreads / 32);
constexpr int kTokChunk = 32;
constexpr int kMaxVPerLane = 16;  // d_v <= 512

__device__ __forceinline__ float e4m3_to_float(uint8_t v)
{
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v), __NV_E4M3);
    return __half2float(__half(h));
}

// One latent cache as the kernel reads it.
struct SimtCache {
    const uint8_t* vals;
    int64_t vps, vts;
    const uint8_t* scs;
    int64_t sps, sts;
    const int32_t* bt;
    int64_t bt_stride;
    int max_pages, page_kv, num_pages;
};

struct SimtParams {
    const __nv_bfloat16* q;
    int num_heads, d_qk, d_v;
    float softmax_scale;
    SimtCache kv;                      // the selected (sparse) entries
    SimtCache swa;                     // the sliding window (vals null: none)
    int window;
    const int32_t* seq_lens;
    const int32_t* cum_q;
    int batch;
    const int32_t* seq_of_row;
    int next_n;
    const int32_t* idx;
    int64_t idx_stride;
    int k;
    const int32_t* topk_lens;
    __nv_bfloat16* out;
    float* lse;
    int32_t* status;
};

// Latent row of logical position s of sequence b: its bytes (and fp32 token
// scale), or null if the block table has no valid page for it.
__device__ __forceinline__ const uint8_t* simt_row(const SimtCache& c, int b, int s, float* tok_scale)
{
    const int lp = s / c.page_kv;
    const int page = lp < c.max_pages ? c.bt[static_cast<int64_t>(b) * c.bt_stride + lp] : -1;
    if (page < 0 || page >= c.num_pages)
        return nullptr;
    if (c.scs)
        *tok_scale = *reinterpret_cast<const float*>(c.scs + page * c.sps + (s % c.page_kv) * c.sts);
    return c.vals + page * c.vps + (s % c.page_kv) * c.vts;
}

template <int kFmt>
__global__ void __launch_bounds__(kThreads)
mla_simt_kernel(const SimtParams p)
{
    extern __shared__ float smf[];
    pdl_wait();                                        // nothing the previous kernel writes is read before
    const int d_qk = p.d_qk, d_v = p.d_v, num_heads = p.num_heads;
    float* q_s = smf;                                  // [kHeadsPerCta][d_qk]
    float* c_s = q_s + kHeadsPerCta * d_qk;            // [kTokChunk][d_qk]
    __shared__ int valid_s[kTokChunk];

    const int r = blockIdx.x;
    const int h0 = blockIdx.y * kHeadsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const MlaRowSeq rs = mla_row_seq(r, p.cum_q, p.batch, p.seq_of_row, p.next_n);
    const int b = rs.seq;
    // this row's token slots: the first kr entries of its index list, then the
    // w window positions [win0, win0 + w)
    int kr = p.k, w = 0, win0 = 0;
    if (b < 0) {
        kr = 0;                                        // a row outside every sequence: no key
        if (threadIdx.x == 0 && blockIdx.y == 0 && p.status)
            atomicOr(p.status, DSA_DEV_BAD_INDEX);
    } else {
        if (p.topk_lens)
            kr = min(max(p.topk_lens[r], 0), p.k);
        if (p.swa.vals) {
            const int vis = visible_len(max(p.seq_lens[b], 0), rs.q_len, rs.i);
            w = min(p.window, vis);
            win0 = vis - w;
        }
    }
    const int nslots = kr + w;

    for (int e = threadIdx.x; e < kHeadsPerCta * d_qk; e += kThreads) {
        const int hh = e / d_qk, d = e % d_qk;
        const int h = h0 + hh;
        q_s[e] = h < num_heads ? __bfloat162float(p.q[(static_cast<int64_t>(r) * num_heads + h) * d_qk + d]) : 0.f;
    }

    float m[kHeadsPerWarp], l[kHeadsPerWarp], o[kHeadsPerWarp][kMaxVPerLane];
#pragma unroll
    for (int a = 0; a < kHeadsPerWarp; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int v = 0; v < kMaxVPerLane; ++v)
            o[a][v] = 0.f;
    }

    const int32_t* irow = p.idx + static_cast<int64_t>(r) * p.idx_stride;
    for (int j0 = 0; j0 < nslots; j0 += kTokChunk) {
        __syncthreads();
        // gather + decode: warp w handles slots w, w+8, ...
        for (int t = warp; t < kTokChunk; t += kThreads / 32) {
            const int j = j0 + t;
            const uint8_t* src = nullptr;
            float tok_scale = 1.f;
            if (j < kr) {
                const int s = irow[j];
                if (s >= 0) {
                    src = simt_row(p.kv, b, s, &tok_scale);
                    if (!src && lane == 0 && p.status)
                        atomicOr(p.status, DSA_DEV_BAD_INDEX);
                }
            } else if (j < nslots) {
                src = simt_row(p.swa, b, win0 + j - kr, &tok_scale);
                if (!src && lane == 0 && p.status)
                    atomicOr(p.status, DSA_DEV_BAD_INDEX);
            }
            if (lane == 0)
                valid_s[t] = src != nullptr;
            if (!src)
                continue;
            for (int d = lane; d < d_qk; d += 32) {
                float v;
                if (kFmt == DSA_KV_FP8_E4M3)
                    v = e4m3_to_float(src[d]) * tok_scale;
                else
                    v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[d]);
                c_s[t * d_qk + d] = v;
            }
        }
        __syncthreads();
        for (int t = 0; t < kTokChunk; ++t) {
            if (!valid_s[t])
                continue;
            const float* c = c_s + t * d_qk;
#pragma unroll
            for (int a = 0; a < kHeadsPerWarp; ++a) {
                const float* qh = q_s + (warp * kHeadsPerWarp + a) * d_qk;
                float dot = 0.f;
                for (int d = lane; d < d_qk; d += 32)
                    dot = fmaf(qh[d], c[d], dot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    dot += __shfl_xor_sync(0xffffffffu, dot, off);
                const float sc = dot * p.softmax_scale;
                const float mn = fmaxf(m[a], sc);
                const float alpha = expf(m[a] - mn);
                const float pj = expf(sc - mn);
                l[a] = l[a] * alpha + pj;
#pragma unroll
                for (int v = 0; v < kMaxVPerLane; ++v) {
                    const int d = lane + 32 * v;
                    if (d < d_v)
                        o[a][v] = fmaf(pj, c[d], o[a][v] * alpha);
                }
                m[a] = mn;
            }
        }
    }

#pragma unroll
    for (int a = 0; a < kHeadsPerWarp; ++a) {
        const int h = h0 + warp * kHeadsPerWarp + a;
        if (h >= num_heads)
            continue;
        const int64_t base = static_cast<int64_t>(r) * num_heads + h;
        const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
#pragma unroll
        for (int v = 0; v < kMaxVPerLane; ++v) {
            const int d = lane + 32 * v;
            if (d < d_v)
                p.out[base * d_v + d] = __float2bfloat16(o[a][v] * inv);
        }
        if (lane == 0)
            p.lse[base] = l[a] > 0.f ? m[a] + logf(l[a]) : -INFINITY;
    }
}

}  // namespace

// Launch as a programmatic dependent of the previous kernel of the stream.
template <class K>
static cudaError_t launch_pdl(K kern, dim3 grid, int smem, cudaStream_t stream, const SimtParams& p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

static SimtCache simt_cache(const dsa_paged_cache* c)
{
    SimtCache s{};
    if (!c)
        return s;
    s.vals = static_cast<const uint8_t*>(c->values);
    s.vps = c->val_page_stride;
    s.vts = c->val_token_stride;
    s.scs = c->fmt == DSA_KV_FP8_E4M3 ? static_cast<const uint8_t*>(c->scales) : nullptr;
    s.sps = c->sc_page_stride;
    s.sts = c->sc_token_stride;
    s.bt = c->block_table;
    s.bt_stride = c->bt_row_stride;
    s.max_pages = c->max_pages_per_seq;
    s.page_kv = c->page_kv;
    s.num_pages = c->num_pages;
    return s;
}

dsa_status launch_sparse_mla_simt(const MlaArgs& a, cudaStream_t stream)
{
    const dsa_paged_cache* kv = a.kv;
    const dim3 grid(a.rows, (a.num_heads + kHeadsPerCta - 1) / kHeadsPerCta);
    const int smem = (kHeadsPerCta + kTokChunk) * a.d_qk * 4;
    if (a.rows == 0)
        return DSA_OK;
    SimtParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.num_heads = a.num_heads;
    p.d_qk = a.d_qk;
    p.d_v = a.d_v;
    p.softmax_scale = a.softmax_scale;
    p.kv = simt_cache(kv);
    p.swa = simt_cache(a.swa);
    p.window = a.swa ? a.window : 0;
    p.seq_lens = a.seq_lens;
    p.cum_q = a.cum_q;
    p.batch = a.batch;
    p.seq_of_row = a.seq_of_row;
    p.next_n = a.next_n;
    p.idx = a.idx;
    p.idx_stride = a.idx_row_stride;
    p.k = a.k;
    p.topk_lens = a.topk_lens;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.status = a.status;
    cudaError_t e;
    if (kv->fmt == DSA_KV_FP8_E4M3) {
        e = cudaFuncSetAttribute(mla_simt_kernel<DSA_KV_FP8_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        e = launch_pdl(mla_simt_kernel<DSA_KV_FP8_E4M3>, grid, smem, stream, p);
    } else {
        e = cudaFuncSetAttribute(mla_simt_kernel<DSA_KV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        e = launch_pdl(mla_simt_kernel<DSA_KV_BF16>, grid, smem, stream, p);
    }
    if (e != cudaSuccess)
        return cuda_fail(e);
    return check_launch();
}

}  // namespace dsa
