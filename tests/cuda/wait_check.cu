// Test helper (built by tests/test_gpu_bounded_wait.py): the bounded mbarrier
// wait of the tensor-core GEMM, driven to its limit on a barrier that nothing
// arrives on.  The kernel returns normally; the host reads what it recorded.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"
#include "tc_ptx.cuh"

namespace {

// out[0]: wait result (1 = phase seen), out[1]: status word after the wait,
// out[2]: elapsed ns.  preset: value written to the status word before the
// wait (another thread's error).
__global__ void wait_kernel(uint64_t limit_ns, int preset, long long* out, int* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    *status = preset;
    const uint32_t b = moe::ptx::smem_addr(&bar);
    moe::ptx::mbar_init(b, 1);
    moe::ptx::fence_barrier_init();
    const uint64_t t0 = moe::ptx::globaltimer();
    // phase 0 never completes: no thread arrives
    const bool ok = moe::ptx::mbar_wait(b, 0, status, limit_ns, MOE_ERR_TIMEOUT);
    out[0] = ok ? 1 : 0;
    out[1] = *reinterpret_cast<volatile int*>(status);
    out[2] = (long long)(moe::ptx::globaltimer() - t0);
}

}  // namespace

extern "C" int wait_check(unsigned long long limit_ns, int preset, long long* host_out) {
    long long* d = nullptr;
    if (cudaMalloc(&d, 3 * sizeof(long long) + sizeof(int)) != cudaSuccess) return 1;
    wait_kernel<<<1, 32>>>(limit_ns, preset, d, reinterpret_cast<int*>(d + 3));
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(host_out, d, 3 * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
