// eplb_collect.cu -- the load-aggregation half of the EPLB loop.
//
// "xDeepServe on CloudMatrix384", section "专家负载均衡", P068: a Collect kernel
// after gating counts the tokens each expert receives; the counts are
// aggregated over a time window and sent, periodically, to the planner
// (P069-P076), whose input is the load of every logical expert in each time
// slice.  moe_route already writes the per-physical-expert counts of one
// step; this kernel folds them into the logical loads of the current slice
// on the device, so a slice costs no host transfer until the window is read.
#include "internal.cuh"

namespace {

// A phys_to_logical entry outside [0, E_log) is caller data that names no
// logical expert: its count is skipped.
__global__ void eplb_collect_kernel(int E_log, int E_phys, const int32_t* __restrict__ expert_counts,
                                    const int32_t* __restrict__ phys_to_logical,
                                    long long* __restrict__ load) {
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < E_phys; p += gridDim.x * blockDim.x) {
        const int e = phys_to_logical ? phys_to_logical[p] : p;
        const int c = expert_counts[p];
        if (c && e >= 0 && e < E_log)
            atomicAdd(reinterpret_cast<unsigned long long*>(load + e), (unsigned long long)c);
    }
}

}  // namespace

extern "C" moe_status moe_eplb_collect(int32_t E_log, int32_t E_phys, const int32_t* expert_counts,
                                       const int32_t* phys_to_logical, int64_t* load,
                                       moe_stream_t stream) {
    if (E_log < 1 || E_phys < E_log || !expert_counts || !load) return MOE_ERR_INVALID_ARG;
    if (!phys_to_logical && E_phys != E_log) return MOE_ERR_INVALID_ARG;
    const int threads = 256;
    const int blocks = (E_phys + threads - 1) / threads;
    eplb_collect_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(
        E_log, E_phys, expert_counts, phys_to_logical, reinterpret_cast<long long*>(load));
    moe::count_launches(1);
    return moe::record_cuda_status(cudaGetLastError());
}
