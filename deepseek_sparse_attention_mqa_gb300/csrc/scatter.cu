// scatter.cu -- quantise new K rows and write them into a paged cache.
//
// "feat(deepseek_v4): Add fp4 indexer for dsv4" (ROCm/ATOM #1709), commit notes:
// the FP4 indexer ships a scatter kernel beside its mqa-logits kernel, which
// writes each new token's K into the paged FP4 cache.  Here the same step
// serves both cache formats of this library, through a slot mapping (slot =
// physical page * page_kv + row, negative = padding token, skipped):
//  - FP8: per token, scale = amax / 448 (fp32; 1 for an all-zero row), codes
//    e4m3(x / scale) rounded to nearest, ties to even, saturating; the fp32
//    scale is stored beside the token.
//  - MXFP4 (OCP MX v1.0): per 32-element block, shared exponent
//    e = floor(log2 amax) - 2 (clamped to [-127, 127]) stored as ue8m0 e + 127;
//    codes e2m1(x * 2^-e), ties to even, saturating at 6, two per byte with the
//    even element in the low nibble.
// Every code's sign bit is the sign bit of the value it encodes.
//
// HBM-bound and tiny: one warp per token, each lane owning 8-element chunks
// (one 16-byte bf16 load or two fp32 loads), the token's or block's amax found
// with warp shuffles, and the codes stored as 8 (FP8) or 4 (MXFP4) bytes per
// lane, so a warp's stores of one row are contiguous.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host.h"

namespace dsa {
namespace {

constexpr int kScatterWarps = 8;

// Nearest e4m3 ("fn") code, ties to the even code, saturating to +-448.
__device__ __forceinline__ uint32_t enc_e4m3(float v)
{
    const uint32_t sign = (__float_as_uint(v) >> 24) & 0x80u;
    const float a = fabsf(v);
    uint32_t code;
    if (!(a < 448.f)) {
        code = 0x7Eu;
    } else if (a < 0.015625f) {                              // below 2^-6: multiples of 2^-9
        code = static_cast<uint32_t>(__float2int_rn(a * 512.f));   // 0 .. 8 (8 is 2^-6, code 0x08)
    } else {
        int E = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu) - 127;   // a in [2^E, 2^(E+1))
        // a * 2^(3-E) lies in [8, 16): its nearest integer is 8 + the 3-bit mantissa
        int m = __float2int_rn(a * __uint_as_float(static_cast<uint32_t>(127 + 3 - E) << 23));
        if (m == 16) {
            m = 8;
            ++E;
        }
        code = static_cast<uint32_t>(((E + 7) << 3) | (m - 8));
    }
    return sign | code;
}

// Nearest e2m1 code (4 bits), ties to the even code, saturating to +-6.
__device__ __forceinline__ uint32_t enc_e2m1(float v)
{
    const uint32_t sign = (__float_as_uint(v) >> 28) & 0x8u;
    const float a = fabsf(v);
    int code;
    if (!(a < 6.f))
        code = 7;
    else if (a < 2.f)
        code = __float2int_rn(a * 2.f);          // 0, 0.5, 1, 1.5, 2 -> codes 0..4
    else if (a < 4.f)
        code = __float2int_rn(a) + 2;            // 2, 3, 4 -> codes 4..6
    else
        code = __float2int_rn(a * 0.5f) + 4;     // 4, 6 -> codes 6, 7
    return sign | static_cast<uint32_t>(code);
}

template <bool kBf16>
__device__ __forceinline__ void load_chunk(const void* k, int64_t row_elems, int c, float (&x)[8])
{
    if constexpr (kBf16) {
        const uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(k) + row_elems + c * 8);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(k) + row_elems + c * 8);
        const float4 a = p[0], b = p[1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
}

struct ScatterParams {
    const void* k;
    int64_t k_stride;           // elements
    int n_tokens;
    int D;
    const int64_t* slots;
    uint8_t* vals;
    int64_t vps, vts;
    uint8_t* scales;
    int64_t sps, sts;
    int page_kv;
    int num_pages;
    int32_t* status;
};

// FP8: one warp per token; chunks c = lane + 32 j of 8 elements.
template <bool kBf16>
__global__ void __launch_bounds__(32 * kScatterWarps)
scatter_fp8_kernel(const ScatterParams p)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
    if (t >= p.n_tokens)
        return;
    const int64_t slot = p.slots[t];
    if (slot < 0)
        return;
    const int64_t page = slot / p.page_kv, row = slot % p.page_kv;
    if (page >= p.num_pages) {
        if (lane == 0 && p.status)
            atomicOr(p.status, DSA_DEV_BAD_PAGE);
        return;
    }
    const int nchunks = p.D / 8;
    const int64_t krow = static_cast<int64_t>(t) * p.k_stride;
    float amax = 0.f;
    // pass 1: the token's amax (the row is re-read from L1/L2 in pass 2)
    for (int c = lane; c < nchunks; c += 32) {
        float x[8];
        load_chunk<kBf16>(p.k, krow, c, x);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint8_t* vrow = p.vals + page * p.vps + row * p.vts;
    for (int c = lane; c < nchunks; c += 32) {
        float x[8];
        load_chunk<kBf16>(p.k, krow, c, x);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo |= enc_e4m3(__fdiv_rn(x[i], scale)) << (8 * i);
            hi |= enc_e4m3(__fdiv_rn(x[4 + i], scale)) << (8 * i);
        }
        *reinterpret_cast<uint2*>(vrow + c * 8) = make_uint2(lo, hi);
    }
    if (lane == 0)
        *reinterpret_cast<float*>(p.scales + page * p.sps + row * p.sts) = scale;
}

// MXFP4: one warp per token; a 32-element block is 4 consecutive chunks, i.e.
// 4 consecutive lanes of one iteration.
template <bool kBf16>
__global__ void __launch_bounds__(32 * kScatterWarps)
scatter_mxfp4_kernel(const ScatterParams p)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
    if (t >= p.n_tokens)
        return;
    const int64_t slot = p.slots[t];
    if (slot < 0)
        return;
    const int64_t page = slot / p.page_kv, row = slot % p.page_kv;
    if (page >= p.num_pages) {
        if (lane == 0 && p.status)
            atomicOr(p.status, DSA_DEV_BAD_PAGE);
        return;
    }
    const int nchunks = p.D / 8;                  // a multiple of 4
    const int64_t krow = static_cast<int64_t>(t) * p.k_stride;
    uint8_t* vrow = p.vals + page * p.vps + row * p.vts;
    uint8_t* srow = p.scales + page * p.sps + row * p.sts;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
        const int c = c0 + lane;
        const bool on = c < nchunks;              // uniform per group of 4 lanes
        float x[8];
        float amax = 0.f;
        if (on) {
            load_chunk<kBf16>(p.k, krow, c, x);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                amax = fmaxf(amax, fabsf(x[i]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // floor(log2 amax) from the exponent field; zero and subnormal amax give
        // an exponent below -127, clamped to -127
        const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
        const int e = ef == 0 ? -127 : max(-127, ef - 127 - 2);          // <= 125
        if (on) {
            const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e
            uint32_t packed = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                packed |= enc_e2m1(x[i] * inv) << (4 * i);
            *reinterpret_cast<uint32_t*>(vrow + c * 4) = packed;
            if ((c & 3) == 0)
                srow[c >> 2] = static_cast<uint8_t>(e + 127);
        }
    }
}

}  // namespace

dsa_status launch_kv_scatter(const void* k, bool bf16, int64_t k_stride, int n_tokens, const int64_t* slots,
                             const dsa_paged_cache* c, int32_t* status, cudaStream_t stream)
{
    ScatterParams p;
    p.k = k;
    p.k_stride = k_stride;
    p.n_tokens = n_tokens;
    p.D = c->head_dim;
    p.slots = slots;
    p.vals = static_cast<uint8_t*>(const_cast<void*>(c->values));
    p.vps = c->val_page_stride;
    p.vts = c->val_token_stride;
    p.scales = static_cast<uint8_t*>(const_cast<void*>(c->scales));
    p.sps = c->sc_page_stride;
    p.sts = c->sc_token_stride;
    p.page_kv = c->page_kv;
    p.num_pages = c->num_pages;
    p.status = status;
    const dim3 grid((n_tokens + kScatterWarps - 1) / kScatterWarps);
    const dim3 block(32 * kScatterWarps);
    if (c->fmt == DSA_KV_FP8_E4M3) {
        if (bf16)
            scatter_fp8_kernel<true><<<grid, block, 0, stream>>>(p);
        else
            scatter_fp8_kernel<false><<<grid, block, 0, stream>>>(p);
    } else {
        if (bf16)
            scatter_mxfp4_kernel<true><<<grid, block, 0, stream>>>(p);
        else
            scatter_mxfp4_kernel<false><<<grid, block, 0, stream>>>(p);
    }
    return check_launch();
}

}  // namespace dsa
