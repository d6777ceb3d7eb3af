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

template <int kFmt>
__global__ void __launch_bounds__(kThreads)
mla_simt_kernel(const __nv_bfloat16* __restrict__ q, int num_heads, int d_qk, int d_v,
                float softmax_scale, const uint8_t* __restrict__ vals, int64_t vps, int64_t vts,
                const uint8_t* __restrict__ scs, int64_t sps, int64_t sts,
                const int32_t* __restrict__ block_table, int64_t bt_stride, int max_pages,
                int page_kv, int num_pages, const int32_t* __restrict__ seq_of_row, int next_n,
                const int32_t* __restrict__ idx, int64_t idx_stride, int k,
                __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int32_t* __restrict__ status)
{
    extern __shared__ float smf[];
    float* q_s = smf;                                  // [kHeadsPerCta][d_qk]
    float* c_s = q_s + kHeadsPerCta * d_qk;            // [kTokChunk][d_qk]
    __shared__ int valid_s[kTokChunk];

    const int r = blockIdx.x;
    const int h0 = blockIdx.y * kHeadsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = seq_of_row ? seq_of_row[r] : r / next_n;

    for (int e = threadIdx.x; e < kHeadsPerCta * d_qk; e += kThreads) {
        const int hh = e / d_qk, d = e % d_qk;
        const int h = h0 + hh;
        q_s[e] = h < num_heads ? __bfloat162float(q[(static_cast<int64_t>(r) * num_heads + h) * d_qk + d]) : 0.f;
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

    const int32_t* irow = idx + static_cast<int64_t>(r) * idx_stride;
    for (int j0 = 0; j0 < k; j0 += kTokChunk) {
        __syncthreads();
        // gather + decode: warp w handles tokens w, w+8, ...
        for (int t = warp; t < kTokChunk; t += kThreads / 32) {
            const int j = j0 + t;
            int s = j < k ? irow[j] : -1;
            int page = -1;
            if (s >= 0) {
                const int lp = s / page_kv;
                if (lp < max_pages)
                    page = block_table[static_cast<int64_t>(b) * bt_stride + lp];
                if (page < 0 || page >= num_pages) {
                    if (lane == 0 && status)
                        atomicOr(status, DSA_DEV_BAD_INDEX);
                    s = -1;
                }
            }
            if (lane == 0)
                valid_s[t] = s >= 0;
            if (s < 0)
                continue;
            const uint8_t* src = vals + page * vps + (s % page_kv) * vts;
            float tok_scale = 1.f;
            if (kFmt == DSA_KV_FP8_E4M3)
                tok_scale = *reinterpret_cast<const float*>(scs + page * sps + (s % page_kv) * sts);
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
                const float sc = dot * softmax_scale;
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
                out[base * d_v + d] = __float2bfloat16(o[a][v] * inv);
        }
        if (lane == 0)
            lse[base] = l[a] > 0.f ? m[a] + logf(l[a]) : -INFINITY;
    }
}

}  // namespace

dsa_status launch_sparse_mla_simt(const MlaArgs& a, cudaStream_t stream)
{
    const dsa_paged_cache* kv = a.kv;
    const dim3 grid(a.rows, (a.num_heads + kHeadsPerCta - 1) / kHeadsPerCta);
    const int smem = (kHeadsPerCta + kTokChunk) * a.d_qk * 4;
    if (a.rows == 0)
        return DSA_OK;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    cudaError_t e;
    if (kv->fmt == DSA_KV_FP8_E4M3) {
        e = cudaFuncSetAttribute(mla_simt_kernel<DSA_KV_FP8_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        mla_simt_kernel<DSA_KV_FP8_E4M3><<<grid, kThreads, smem, stream>>>(
            q, a.num_heads, a.d_qk, a.d_v, a.softmax_scale, static_cast<const uint8_t*>(kv->values),
            kv->val_page_stride, kv->val_token_stride, static_cast<const uint8_t*>(kv->scales), kv->sc_page_stride,
            kv->sc_token_stride, kv->block_table, kv->bt_row_stride, kv->max_pages_per_seq, kv->page_kv,
            kv->num_pages, a.seq_of_row, a.next_n, a.idx, a.idx_row_stride, a.k, out, a.lse, a.status);
    } else {
        e = cudaFuncSetAttribute(mla_simt_kernel<DSA_KV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return cuda_fail(e);
        mla_simt_kernel<DSA_KV_BF16><<<grid, kThreads, smem, stream>>>(
            q, a.num_heads, a.d_qk, a.d_v, a.softmax_scale, static_cast<const uint8_t*>(kv->values),
            kv->val_page_stride, kv->val_token_stride, nullptr, 0, 0, kv->block_table, kv->bt_row_stride,
            kv->max_pages_per_seq, kv->page_kv, kv->num_pages, a.seq_of_row, a.next_n, a.idx,
            a.idx_row_stride, a.k, out, a.lse, a.status);
    }
    return check_launch();
}

}  // namespace dsa
