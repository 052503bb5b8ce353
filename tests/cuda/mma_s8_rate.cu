// mma_s8_rate.cu -- rate of the legacy warp-level INT8 tensor-core MMA
// (mma.sync m16n8k32, s8 x s8 -> s32) on sm_103a.
//
// sm_103a has no INT8 kind of tcgen05.mma, so the exact int8 contraction of
// the expert FFN runs on the fp16 kind of tcgen05.  The only other INT8
// tensor-core instruction left on this target is the warp-level mma.sync;
// this program measures how fast it can go, so the expert GEMM's rate can be
// set against both.
//
// Every warp keeps kChains independent accumulator fragments in registers
// and issues kChains MMAs per iteration on constant operand fragments (every
// int8 byte = a for A, b for B).  After `iters` iterations every accumulator
// element equals iters * 32 * a * b, which the host checks: a result that is
// not that value means the timed loop did not do the work.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kChains = 8;

__global__ void __launch_bounds__(256) mma_s8_loop(int iters, int a_val, int b_val, int* out) {
    const uint32_t a = (uint32_t)(a_val & 0xff) * 0x01010101u;
    const uint32_t b = (uint32_t)(b_val & 0xff) * 0x01010101u;
    int c[kChains][4];
#pragma unroll
    for (int j = 0; j < kChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a), "r"(a), "r"(a), "r"(a), "r"(b), "r"(b));
        }
    }
    // every element must hold the same value; report it, or INT32_MIN if any differs
    int v = c[0][0];
    bool same = true;
#pragma unroll
    for (int j = 0; j < kChains; ++j)
        same = same && c[j][0] == v && c[j][1] == v && c[j][2] == v && c[j][3] == v;
    out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = same ? v : INT32_MIN;
}

}  // namespace

extern "C" {

// Runs `reps` timed launches of `blocks` x 256 threads after one warm-up
// launch.  out (device, blocks*256 ints) receives every thread's accumulator
// value from the last launch.  *ms = mean duration of one launch (CUDA events);
// *ops = integer operations (2 per multiply-add) of one launch.
int mma_s8_rate(int blocks, int iters, int reps, int a_val, int b_val, int* out, float* ms,
                double* ops) {
    if (blocks <= 0 || iters <= 0 || reps <= 0 || !out || !ms || !ops) return 1;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return 2;
    mma_s8_loop<<<blocks, 256>>>(iters, a_val, b_val, out);
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r) mma_s8_loop<<<blocks, 256>>>(iters, a_val, b_val, out);
    cudaEventRecord(e1);
    cudaError_t err = cudaEventSynchronize(e1);
    float t = 0.f;
    cudaEventElapsedTime(&t, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return 3;
    *ms = t / reps;
    // per warp and iteration: kChains MMAs of 16 x 8 x 32 multiply-adds
    *ops = (double)blocks * 8 * (double)iters * kChains * 2.0 * 16 * 8 * 32;
    return 0;
}

}  // extern "C"
