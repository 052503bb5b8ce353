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
// route-slot order.  A NaN logit is read as -inf, so every selected id is a
// valid expert whatever the logits hold.
// Counts (count_kernel): no atomics.  One cluster of kCountBlocks blocks;
// each warp counts its share of the T*k physical ids into a histogram row of
// its own in shared memory (the lanes holding the same id elect their lowest
// lane with match_any, which adds the group's size, so no two lanes write one
// word); each block sums its warps' rows; after a cluster barrier, block b
// sums its range of experts over the blocks' totals through distributed
// shared memory and writes them.
#include <cooperative_groups.h>

#include "internal.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kCountBlocks = 8;      // one cluster (portable size)
constexpr int kCountThreads = 1024;
constexpr int kCountWarps = kCountThreads / 32;
constexpr int kCountUnroll = 4;      // id loads in flight per lane

__device__ __forceinline__ bool better(float v, int id, float bv, int bid) {
    return v > bv || (v == bv && id < bid);
}

template <int VPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_kernel(int T, int E, int E_phys, int k, const float* __restrict__ logits,
             const int32_t* __restrict__ rep_table, const int32_t* __restrict__ n_copies,
             int max_copies, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
             int32_t* __restrict__ phys_idx) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t < T) {
        const float* lrow = logits + (long long)t * E;
        float v[VPL];
        unsigned taken = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            int e = lane + 32 * i;
            const float l = e < E ? __ldg(lrow + e) : -INFINITY;
            v[i] = isnan(l) ? -INFINITY : l;
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
                // n_copies and rep_table entries are caller data: an entry
                // outside its range gives -1 (not counted; the dispatch
                // reports it) and is never used as an address
                const int nc = n_copies[my_id];
                p = -1;
                if (nc >= 1 && nc <= max_copies) {
                    p = rep_table[(long long)my_id * max_copies + (t % nc)];
                    if (p < 0 || p >= E_phys) p = -1;
                }
            }
            phys_idx[o] = p;
        }
    }
}

__global__ void __cluster_dims__(kCountBlocks, 1, 1) __launch_bounds__(kCountThreads)
count_kernel(long long n, int E_phys, const int32_t* __restrict__ phys_idx,
             int32_t* __restrict__ expert_counts) {
    extern __shared__ int s_cnt[];  // [kCountWarps][E_phys]; row 0 ends as the block's totals
    cg::cluster_group cluster = cg::this_cluster();
    const int b = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kCountWarps * E_phys; i += kCountThreads) s_cnt[i] = 0;
    __syncthreads();
    // this block's contiguous share of the ids in rounds of 32; warp w takes
    // rounds w, w + 32, ..., loading kCountUnroll rounds before counting them
    const long long per = (n + kCountBlocks - 1) / kCountBlocks;
    const long long lo = (long long)b * per, hi = min(n, lo + per);
    const long long rounds = hi > lo ? (hi - lo + 31) / 32 : 0;
    const unsigned lt = (1u << lane) - 1u;
    int* row = s_cnt + warp * E_phys;
    for (long long r0 = warp; r0 < rounds; r0 += (long long)kCountWarps * kCountUnroll) {
        int p[kCountUnroll];
#pragma unroll
        for (int u = 0; u < kCountUnroll; ++u) {
            const long long i = lo + (r0 + (long long)u * kCountWarps) * 32 + lane;
            p[u] = i < hi ? __ldg(phys_idx + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kCountUnroll; ++u) {
            const int q = (p[u] >= 0 && p[u] < E_phys) ? p[u] : -1;  // -1: invalid route, not counted
            const unsigned same = __match_any_sync(0xffffffffu, q);
            if (q >= 0 && (same & lt) == 0) row[q] += __popc(same);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E_phys; e += kCountThreads) {
        int c = 0;
#pragma unroll 8
        for (int w = 0; w < kCountWarps; ++w) c += s_cnt[w * E_phys + e];
        s_cnt[e] = c;
    }
    cluster.sync();  // every block's totals are final
    const int chunk = (E_phys + kCountBlocks - 1) / kCountBlocks;
    for (int e = b * chunk + threadIdx.x; e < min(E_phys, (b + 1) * chunk); e += kCountThreads) {
        int c = 0;
#pragma unroll
        for (int r = 0; r < kCountBlocks; ++r) c += cluster.map_shared_rank(s_cnt, r)[e];
        expert_counts[e] = c;
    }
    cluster.sync();  // no block leaves while another still reads its shared memory
}

}  // namespace

cudaError_t launch_route(const Dims& d, const float* logits, const int32_t* rep_table,
                         const int32_t* n_copies, int max_copies, int32_t* topk_idx,
                         float* topk_w, int32_t* phys_idx, int32_t* expert_counts,
                         cudaStream_t st) {
    dim3 grid((d.T + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
    int vpl = (d.E_log + 31) / 32;
#define MOE_ROUTE_CASE(V)                                                                  \
    route_kernel<V><<<grid, block, 0, st>>>(d.T, d.E_log, d.E_phys, d.k, logits,           \
                                            rep_table, n_copies, max_copies, topk_idx,     \
                                            topk_w, phys_idx)
    if (vpl <= 1) MOE_ROUTE_CASE(1);
    else if (vpl <= 2) MOE_ROUTE_CASE(2);
    else if (vpl <= 4) MOE_ROUTE_CASE(4);
    else if (vpl <= 8) MOE_ROUTE_CASE(8);
    else if (vpl <= 16) MOE_ROUTE_CASE(16);
    else MOE_ROUTE_CASE(32);
#undef MOE_ROUTE_CASE
    const size_t smem = sizeof(int) * (size_t)kCountWarps * d.E_phys;
    cudaError_t e = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    count_kernel<<<kCountBlocks, kCountThreads, smem, st>>>((long long)d.T * d.k, d.E_phys, phys_idx,
                                                            expert_counts);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace moe
