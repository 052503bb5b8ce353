// Test helper (built by tests/test_gpu_device_math.py) for the library's
// device arithmetic:
//   - the expert-FFN SiLU, straightforward form (silu_spec, IEEE division)
//     against the branch-free form (silu_fast) of the gate/up GEMM epilogue;
//   - token-wise INT8 codes, IEEE-division form (quant1) against the
//     reciprocal form with Markstein's correction (quant_row_n, one value and
//     groups of 16) of the dispatch and requantisation kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"

namespace {

__global__ void compare_all(unsigned long long* mismatches, unsigned* first_bad) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned long long bad = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (1ull << 32); i += stride) {
        const float g = __uint_as_float((uint32_t)i);
        const float a = moe::silu_spec(g), b = moe::silu_fast(g);
        const bool same = (__float_as_uint(a) == __float_as_uint(b)) || (isnan(a) && isnan(b));
        if (!same) {
            ++bad;
            atomicMin(first_bad, (unsigned)i);
        }
    }
    if (bad) atomicAdd(mismatches, bad);
}

__global__ void eval(const float* in, float* spec, float* fast, float* ex, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        spec[i] = moe::silu_spec(in[i]);
        fast[i] = moe::silu_fast(in[i]);
        ex[i] = moe::exp_spec(in[i]);
    }
}

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16; x *= 0x7feb352du; x ^= x >> 15; x *= 0x846ca68bu; x ^= x >> 16;
    return x;
}

// n random (row absmax a, value v) pairs with |v| <= a: a spans binades
// 2^-120 .. 2^120 (plus the smallest normal scales); half of the v lie within
// 4 ulp of (c + 1/2) * s for a random integer c, where the two forms could
// round differently.
__global__ void compare_quant(unsigned long long n, unsigned long long* mismatches,
                              unsigned long long* near_half, unsigned* first_bad) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned long long bad = 0, nh = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t h1 = mix32((uint32_t)i * 2u + 1u), h2 = mix32((uint32_t)(i >> 31) ^ ((uint32_t)i * 2u + 2u) ^ 0x9e3779b9u);
        const int e = (int)(h1 >> 23) % 250 - 125;  // 2^-125 .. 2^124
        const float a = ldexpf(1.0f + (float)(h1 & 0x7fffffu) * 0x1p-23f, e);
        const float s = moe::row_scale(a);
        if (s == 0.f) continue;
        const float rs = moe::quant_rcp(s);
        float v;
        if (h2 & 1u) {
            const int c = (int)((h2 >> 1) % 254u) - 127;
            v = __fmul_rn((float)c + 0.5f, s);
            const int d = (int)((h2 >> 9) % 9u) - 4;
            v = __int_as_float(__float_as_int(v) + d);
            ++nh;
        } else {
            v = __fmul_rn(a, (float)(h2 >> 1) * 0x1p-30f - 1.0f);
        }
        if (!(fabsf(v) <= a)) continue;
        const float v1[1] = {v};
        int q1[1];
        moe::quant_row_n<1>(v1, s, rs, q1);
        if (q1[0] != moe::quant1(v, s)) {
            ++bad;
            atomicMin(first_bad, (unsigned)i);
        }
    }
    if (bad) atomicAdd(mismatches, bad);
    atomicAdd(near_half, nh);
}

// n random rows of 16 values (absmax a as above, each value next to a
// half-integer quotient with probability 1/8, else uniform in [-a, a]):
// quant_row_n<16> of the row against quant1 of each value.  Counts the rows
// holding a value drawn next to a half-integer quotient.
__global__ void compare_quant_rows(unsigned long long n, unsigned long long* mismatches,
                                   unsigned long long* slow_rows, unsigned* first_bad) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned long long bad = 0, ns = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t h1 = mix32((uint32_t)i * 2u + 0x51ed27u);
        const int ex = (int)(h1 >> 23) % 250 - 125;
        const float a = ldexpf(1.0f + (float)(h1 & 0x7fffffu) * 0x1p-23f, ex);
        const float s = moe::row_scale(a);
        if (s == 0.f) continue;
        const float rs = moe::quant_rcp(s);
        float v[16];
        bool near_any = false;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t h2 = mix32(h1 ^ (uint32_t)(i >> 32) ^ (0x9e3779b9u * (uint32_t)(e + 1)));
            float x;
            if ((h2 & 7u) == 0u) {
                const int c = (int)((h2 >> 3) % 254u) - 127;
                x = __fmul_rn((float)c + 0.5f, s);
                const int d = (int)((h2 >> 11) % 9u) - 4;
                x = __int_as_float(__float_as_int(x) + d);
                near_any = true;
            } else {
                x = __fmul_rn(a, (float)(h2 >> 1) * 0x1p-30f - 1.0f);
            }
            v[e] = fabsf(x) <= a ? x : 0.0f;
        }
        int q[16];
        moe::quant_row_n<16>(v, s, rs, q);
        bool row_bad = false;
#pragma unroll
        for (int e = 0; e < 16; ++e) row_bad |= q[e] != moe::quant1(v[e], s);
        if (row_bad) {
            ++bad;
            atomicMin(first_bad, (unsigned)i);
        }
        ns += near_any;
    }
    if (bad) atomicAdd(mismatches, bad);
    atomicAdd(slow_rows, ns);
}

}  // namespace

// Rows (of n random 16-value rows) whose quant_row_n<16> codes differ from
// quant1's, and how many rows held a value drawn next to a half-integer.
extern "C" int quant_rows_check(unsigned long long n, unsigned long long* mismatches,
                                unsigned long long* near_rows, unsigned* first_bad) {
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, 3 * sizeof(unsigned long long)) != cudaSuccess) return 1;
    cudaMemset(d, 0, 2 * sizeof(unsigned long long));
    cudaMemset(d + 2, 0xff, sizeof(unsigned long long));
    compare_quant_rows<<<152 * 8, 256>>>(n, d, d + 1, reinterpret_cast<unsigned*>(d + 2));
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(mismatches, d, sizeof(*d), cudaMemcpyDeviceToHost);
    cudaMemcpy(near_rows, d + 1, sizeof(*d), cudaMemcpyDeviceToHost);
    cudaMemcpy(first_bad, d + 2, sizeof(unsigned), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}

// Mismatching codes among n random (absmax, value) pairs, and how many of the
// pairs were drawn next to a half-integer quotient.
extern "C" int quant_check(unsigned long long n, unsigned long long* mismatches,
                           unsigned long long* near_half, unsigned* first_bad) {
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, 3 * sizeof(unsigned long long)) != cudaSuccess) return 1;
    cudaMemset(d, 0, 2 * sizeof(unsigned long long));
    cudaMemset(d + 2, 0xff, sizeof(unsigned long long));
    compare_quant<<<152 * 8, 256>>>(n, d, d + 1, reinterpret_cast<unsigned*>(d + 2));
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(mismatches, d, sizeof(*d), cudaMemcpyDeviceToHost);
    cudaMemcpy(near_half, d + 1, sizeof(*d), cudaMemcpyDeviceToHost);
    cudaMemcpy(first_bad, d + 2, sizeof(unsigned), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}

// Number of the 2^32 binary32 inputs on which the two forms differ (bitwise;
// any two NaNs count as equal), and the smallest such bit pattern.
extern "C" int silu_check_all(unsigned long long* mismatches, unsigned* first_bad) {
    unsigned long long* d_m = nullptr;
    unsigned* d_f = nullptr;
    if (cudaMalloc(&d_m, sizeof(*d_m)) != cudaSuccess) return 1;
    if (cudaMalloc(&d_f, sizeof(*d_f)) != cudaSuccess) return 1;
    cudaMemset(d_m, 0, sizeof(*d_m));
    cudaMemset(d_f, 0xff, sizeof(*d_f));
    compare_all<<<152 * 8, 256>>>(d_m, d_f);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(mismatches, d_m, sizeof(*d_m), cudaMemcpyDeviceToHost);
    cudaMemcpy(first_bad, d_f, sizeof(*d_f), cudaMemcpyDeviceToHost);
    cudaFree(d_m);
    cudaFree(d_f);
    return e == cudaSuccess ? 0 : 2;
}

// silu_spec, silu_fast and exp_spec of n host inputs.
extern "C" int silu_eval(const float* in, float* spec, float* fast, float* ex, int n) {
    float* d = nullptr;
    if (cudaMalloc(&d, 4ull * sizeof(float) * n) != cudaSuccess) return 1;
    cudaMemcpy(d, in, sizeof(float) * n, cudaMemcpyHostToDevice);
    eval<<<(n + 255) / 256, 256>>>(d, d + n, d + 2ll * n, d + 3ll * n, n);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(spec, d + n, sizeof(float) * n, cudaMemcpyDeviceToHost);
    cudaMemcpy(fast, d + 2ll * n, sizeof(float) * n, cudaMemcpyDeviceToHost);
    cudaMemcpy(ex, d + 3ll * n, sizeof(float) * n, cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
