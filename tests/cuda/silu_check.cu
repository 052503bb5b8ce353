// Test helper (built by tests/test_gpu_silu_exhaustive.py): evaluates the
// expert-FFN SiLU of the library's device code, the straightforward form
// (silu_spec, IEEE division) and the branch-free form (silu_fast) used in the
// gate/up GEMM epilogue.
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

}  // namespace

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
