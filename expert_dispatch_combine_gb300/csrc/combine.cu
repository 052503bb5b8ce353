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
// expert FFN.  One block per token; each thread owns 16 consecutive hidden
// elements at a time, reads them from the k messages (16-byte code loads or
// 32-byte bf16 loads, all issued before the arithmetic), accumulates in
// binary32 in ascending route slot (product and sum rounded separately) and
// stores 16 bf16 values (32 bytes).
#include <cuda_bf16.h>

#include "combine_math.cuh"
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;

// One block per token.  Each thread owns 16 consecutive hidden elements at a
// time and loads them from the first kUnroll messages before any arithmetic
// (k 16-byte or 32-byte loads in flight per thread); messages beyond
// kUnroll follow one at a time.  Accumulation is in ascending route slot.
template <bool kInt8>
__global__ void __launch_bounds__(kCombineThreads, kInt8 ? 6 : 4)
combine_kernel(int H, int k, long long crow, const unsigned char* __restrict__ cbuf,
               const float* __restrict__ cscale, const float* __restrict__ topk_w,
               uint16_t* __restrict__ out) {
    constexpr int kUnroll = 8;
    const int t = blockIdx.x;
    const long long tk = (long long)t * k;
    // every thread reads the first kUnroll gate weights and message scales
    // itself (the same words for the whole block, served by L1): no barrier
    // holds the message loads back behind them
    float w_r[kUnroll], s_r[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
        w_r[j] = j < k ? __ldg(topk_w + tk + j) : 0.f;
        s_r[j] = (kInt8 && j < k) ? __ldg(cscale + tk + j) : 0.f;
    }
    const int nch = H / 16;
    const unsigned char* rows = cbuf + tk * crow;
    uint4* orow = reinterpret_cast<uint4*>(out + (long long)t * H);
    for (int c = threadIdx.x; c < nch; c += kCombineThreads) {
        uint4 q[kUnroll][2];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j)
            if (j < k) load16<kInt8>(rows + j * crow, c, q[j]);
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < kUnroll; ++j)
            if (j < k) accumulate16<kInt8>(q[j], w_r[j], s_r[j], acc);
        for (int j = kUnroll; j < k; ++j) {
            uint4 r[2];
            load16<kInt8>(rows + j * crow, c, r);
            accumulate16<kInt8>(r, __ldg(topk_w + tk + j), kInt8 ? __ldg(cscale + tk + j) : 0.f, acc);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 o;
            o.x = pack_bf16x2(acc[8 * h + 0], acc[8 * h + 1]);
            o.y = pack_bf16x2(acc[8 * h + 2], acc[8 * h + 3]);
            o.z = pack_bf16x2(acc[8 * h + 4], acc[8 * h + 5]);
            o.w = pack_bf16x2(acc[8 * h + 6], acc[8 * h + 7]);
            orow[2 * c + h] = o;
        }
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
