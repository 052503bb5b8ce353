// route.cu -- gate top-k routing (one warp per token).
//
// "xDeepServe on CloudMatrix384", section "合设 MoE-Attention 的 All-to-All"
// (P038: every token goes to its top-k experts by gating score; routing index
// and weight matrices I, W of shape B x k), section "专家负载均衡" (P068 Collect
// kernel counting tokens per expert; P078-P079 logical->physical map,
// physical(i, e) = R_e[i mod |R_e|]).
//
// Each lane holds VPL logits (lane + 32*v); k rounds of a warp-wide arg-max
// with the key (logit descending, expert id ascending) select the experts in
// route-slot order.  Counts: a shared-memory histogram per block, then one
// global atomicAdd per non-empty bin (integer sums, order independent).
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ bool better(float v, int id, float bv, int bid) {
    return v > bv || (v == bv && id < bid);
}

template <int VPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_kernel(int T, int E, int E_phys, int k, const float* __restrict__ logits,
             const int32_t* __restrict__ rep_table, const int32_t* __restrict__ n_copies,
             int max_copies, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
             int32_t* __restrict__ phys_idx, int32_t* __restrict__ expert_counts) {
    extern __shared__ int s_hist[];
    for (int i = threadIdx.x; i < E_phys; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t < T) {
        const float* lrow = logits + (long long)t * E;
        float v[VPL];
        unsigned taken = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            int e = lane + 32 * i;
            v[i] = e < E ? __ldg(lrow + e) : -INFINITY;
            if (e >= E) taken |= 1u << i;  // padding never selected
        }
        int my_id = 0;        // lane j keeps the j-th winner
        float my_val = 0.f;
        float top_val = 0.f;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bid = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                int e = lane + 32 * i;
                if (!(taken & (1u << i)) && better(v[i], e, bv, bid)) { bv = v[i]; bid = e; }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                int oid = __shfl_xor_sync(0xffffffffu, bid, off);
                if (better(ov, oid, bv, bid)) { bv = ov; bid = oid; }
            }
            if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
            if (lane == j) { my_id = bid; my_val = bv; }
            if (j == 0) top_val = bv;
        }
        // renormalised softmax over the k winners
        float z = lane < k ? expf(my_val - top_val) : 0.f;
        float sum = z;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane < k) {
            long long o = (long long)t * k + lane;
            topk_idx[o] = my_id;
            topk_w[o] = z / sum;
            int p = my_id;
            if (rep_table) {
                // n_copies and rep_table entries are caller data: keep every
                // access in bounds (an invalid entry maps to the primary id).
                int nc = min(max(n_copies[my_id], 1), max_copies);
                p = rep_table[(long long)my_id * max_copies + (t % nc)];
                if (p < 0 || p >= E_phys) p = my_id;
            }
            phys_idx[o] = p;
            atomicAdd(&s_hist[p], 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E_phys; i += blockDim.x) {
        int c = s_hist[i];
        if (c) atomicAdd(&expert_counts[i], c);
    }
}

}  // namespace

cudaError_t launch_route(const Dims& d, const float* logits, const int32_t* rep_table,
                         const int32_t* n_copies, int max_copies, int32_t* topk_idx,
                         float* topk_w, int32_t* phys_idx, int32_t* expert_counts,
                         cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * d.E_phys, st);
    if (e != cudaSuccess) return e;
    dim3 grid((d.T + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
    size_t smem = sizeof(int) * d.E_phys;
    int vpl = (d.E_log + 31) / 32;
#define MOE_ROUTE_CASE(V)                                                                  \
    route_kernel<V><<<grid, block, smem, st>>>(d.T, d.E_log, d.E_phys, d.k, logits,        \
                                               rep_table, n_copies, max_copies, topk_idx,  \
                                               topk_w, phys_idx, expert_counts)
    if (vpl <= 1) MOE_ROUTE_CASE(1);
    else if (vpl <= 2) MOE_ROUTE_CASE(2);
    else if (vpl <= 4) MOE_ROUTE_CASE(4);
    else if (vpl <= 8) MOE_ROUTE_CASE(8);
    else if (vpl <= 16) MOE_ROUTE_CASE(16);
    else MOE_ROUTE_CASE(32);
#undef MOE_ROUTE_CASE
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace moe
