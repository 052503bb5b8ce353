// combine_math.cuh -- the FusedCombine arithmetic on 16 hidden elements,
// shared by the combine kernel and the fused return-message/combine path so
// that both round identically: each message value is dequantised (code *
// scale, one binary32 rounding) or widened (bf16), multiplied by the gate
// weight and added in ascending route slot, one rounding per operation.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ float s8_to_f(unsigned w, int b) {
    return (float)(int)(signed char)((w >> (8 * b)) & 0xffu);
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
    return (unsigned)__bfloat16_as_ushort(a) | ((unsigned)__bfloat16_as_ushort(b) << 16);
}

// The raw 16 consecutive hidden elements of a route message (16 codes or 16
// bf16 values).  Messages written earlier in the same kernel by other blocks
// must be read with kCoherent (L2 loads); otherwise the read-only path.
template <bool kInt8, bool kCoherent = false>
__device__ __forceinline__ void load16(const unsigned char* __restrict__ row, int c, uint4 (&q)[2]) {
    const uint4* p = reinterpret_cast<const uint4*>(row);
    if (kInt8) {
        q[0] = kCoherent ? __ldcg(p + c) : __ldg(p + c);
    } else {
        q[0] = kCoherent ? __ldcg(p + 2 * c) : __ldg(p + 2 * c);
        q[1] = kCoherent ? __ldcg(p + 2 * c + 1) : __ldg(p + 2 * c + 1);
    }
}

template <bool kInt8>
__device__ __forceinline__ void accumulate16(const uint4 (&q)[2], float w, float s, float (&acc)[16]) {
    float v[16];
    if (kInt8) {
        const unsigned u[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) v[4 * i + b] = __fmul_rn(s8_to_f(u[i], b), s);
    } else {
        const unsigned u[8] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(u[i] << 16);
            v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(w, v[i]));
}

}  // namespace moe
