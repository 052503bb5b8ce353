// combine_math.cuh -- the FusedCombine arithmetic on 16 hidden elements,
// shared by the combine kernel and the fused return-message/combine path so
// that both round identically.  Messages are taken in ascending route slot;
// a bf16 value is widened, multiplied by the gate weight and added (product
// and sum rounded separately); an INT8 code q with message scale s adds
// RN(w s) * q in one fused multiply-add.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// The four signed bytes of w as binary32, exactly, without integer-to-float
// conversions: with u = q + 128 (the byte xor 0x80), the bit pattern
// 0x4B0000uu is the binary32 value 2^23 + u, and subtracting 2^23 + 128
// leaves q (every step exact).
__device__ __forceinline__ void s8x4_to_f32x4(unsigned w, float (&f)[4]) {
    const unsigned x = w ^ 0x80808080u;
    f[0] = __fsub_rn(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)), 8388736.0f);
    f[1] = __fsub_rn(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541)), 8388736.0f);
    f[2] = __fsub_rn(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542)), 8388736.0f);
    f[3] = __fsub_rn(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543)), 8388736.0f);
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
    if (kInt8) {
        // INT8: the message's factor w * s once, then one fused multiply-add
        // per code (acc + RN(w s) * q, one rounding)
        const float ws = __fmul_rn(w, s);
        const unsigned u[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float f[4];
            s8x4_to_f32x4(u[i], f);
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[4 * i + b] = __fmaf_rn(ws, f[b], acc[4 * i + b]);
        }
    } else {
        const unsigned u[8] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(u[i] << 16);
            v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(w, v[i]));
    }
}

}  // namespace moe
