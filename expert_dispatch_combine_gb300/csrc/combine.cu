// combine.cu -- FusedCombine: dequantise the k return messages of a token and
// take their gate-weighted sum.
//
// "CloudMatrix384 LLM Serving", section "EP320：token 去找专家" (fused_moe
// listing: results are written back by (source_rank, batch_slot, route_slot);
// once all of a token's contributions are in, dequantise and sum them with
// the gate weights).  "xDeepServe on CloudMatrix384", section "合设 MoE-Attention
// 的 All-to-All" (COMBINE procedure: result[token] += value * gate_weight).
//
// On one GPU "all contributions are in" is the kernel boundary after the
// expert FFN.  One block per token; each thread owns 8 consecutive hidden
// elements at a time, reads them from the k messages (8-byte code loads or
// 16-byte bf16 loads), accumulates in binary32 in ascending route slot
// (product and sum rounded separately) and stores 8 bf16 values (16 bytes).
#include <cuda_bf16.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kMaxK = 32;

__device__ __forceinline__ float s8_to_f(unsigned w, int b) {
    return (float)(int)(signed char)((w >> (8 * b)) & 0xffu);
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
    return (unsigned)__bfloat16_as_ushort(a) | ((unsigned)__bfloat16_as_ushort(b) << 16);
}

template <bool kInt8>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(int H, int k, long long crow, const unsigned char* __restrict__ cbuf,
               const float* __restrict__ cscale, const float* __restrict__ topk_w,
               uint16_t* __restrict__ out) {
    __shared__ float s_w[kMaxK], s_s[kMaxK];
    const int t = blockIdx.x;
    const long long tk = (long long)t * k;
    if (threadIdx.x < k) {
        s_w[threadIdx.x] = topk_w[tk + threadIdx.x];
        s_s[threadIdx.x] = kInt8 ? cscale[tk + threadIdx.x] : 0.f;
    }
    __syncthreads();
    const int nch = H / 8;
    uint4* orow = reinterpret_cast<uint4*>(out + (long long)t * H);
    for (int c = threadIdx.x; c < nch; c += kCombineThreads) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const unsigned char* row = cbuf + (tk + j) * crow;
            const float w = s_w[j];
            float v[8];
            if (kInt8) {
                uint2 q = __ldg(reinterpret_cast<const uint2*>(row) + c);
                const float s = s_s[j];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    v[b] = __fmul_rn(s8_to_f(q.x, b), s);
                    v[4 + b] = __fmul_rn(s8_to_f(q.y, b), s);
                }
            } else {
                uint4 q = __ldg(reinterpret_cast<const uint4*>(row) + c);
                v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
                v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
                v[4] = __uint_as_float(q.z << 16); v[5] = __uint_as_float(q.z & 0xffff0000u);
                v[6] = __uint_as_float(q.w << 16); v[7] = __uint_as_float(q.w & 0xffff0000u);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(w, v[i]));
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        orow[c] = o;
    }
}

}  // namespace

cudaError_t launch_combine(const Dims& d, const void* cbuf, long long scale_off,
                           const float* topk_w, uint16_t* out, cudaStream_t st) {
    const unsigned char* cb = static_cast<const unsigned char*>(cbuf);
    if (d.cfmt == MOE_MSG_INT8)
        combine_kernel<true><<<d.T, kCombineThreads, 0, st>>>(
            d.H, d.k, d.crow, cb, reinterpret_cast<const float*>(cb + scale_off), topk_w, out);
    else
        combine_kernel<false><<<d.T, kCombineThreads, 0, st>>>(d.H, d.k, d.crow, cb, nullptr,
                                                                topk_w, out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
