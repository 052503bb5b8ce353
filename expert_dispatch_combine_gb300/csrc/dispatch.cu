// dispatch.cu -- FusedDispatch: token-wise INT8 quantisation fused with the
// scatter of one message per (token, route) into static per-rank buffers.
//
// "CloudMatrix384 LLM Serving", section "EP320：token 去找专家" (fused_moe
// listing: quantise the bf16 row once, then per route_slot write
// {q_token, scale, source_rank, batch_slot, route_slot} into the owner rank's
// static buffer and count the messages per target) and section "缓冲区公式"
// (max_tokens = local_batch * min(topK, experts_per_die)).
// "xDeepServe on CloudMatrix384", section "合设 MoE-Attention 的 All-to-All"
// (P039-P040: per-source counts, prefix sums give each source's place in the
// receiver's area; token-wise INT8 quantisation in the dispatch kernel).
//
// Three kernels:
//   layout_src     one block per source rank: an ordered multi-split of the
//                  rank's lb*k messages by destination rank and by physical
//                  expert (warp match_any + popc, an exclusive scan across
//                  warps) -> slot within (dst, src), rank within (src, expert),
//                  rank_counts[dst][src], hist[src][expert].  No atomics.
//                  A physical id outside [0, E_phys) drops its message
//                  (MOE_ERR_INDEX); a message whose slot would reach
//                  max_tokens (only a replica table mapping two routes of one
//                  token onto one expert can cause it) is marked -1 and
//                  dropped (MOE_ERR_CAPACITY).
//   layout_expert  one block: per-expert prefix over sources and over experts
//                  -> src_base, expert_offsets.
//   scatter        one block per token: bf16 row -> shared memory, absmax,
//                  codes into shared memory, then k bulk asynchronous copies
//                  (shared -> global) of the code row into the k slots, plus
//                  the 16-byte metadata and the expert row list entries.
#include <algorithm>
#include <cuda_fp16.h>

#include "device_math.cuh"
#include "internal.cuh"

namespace moe {
namespace {

// Up to kLayoutMaxWarps warps per source rank, each taking a contiguous run
// of 32-message rounds, so a source's lb*k messages take a few rounds per warp.
constexpr int kLayoutMaxWarps = 16;

__global__ void __launch_bounds__(kLayoutMaxWarps * 32)
layout_src_kernel(int lb, int k, int epr, int R, int E_phys, int S, int mt,
                  const int32_t* __restrict__ phys_idx, int32_t* __restrict__ slot_local,
                  int32_t* __restrict__ erank, int32_t* __restrict__ rank_counts,
                  int32_t* __restrict__ hist, int* __restrict__ err) {
    extern __shared__ int smem[];
    const int W = blockDim.x >> 5;
    int* cntD = smem;                // [W][R]
    int* cntE = cntD + W * R;        // [W][E_phys]
    int* totD = cntE + W * E_phys;   // [R]
    int* totE = totD + R;                      // [E_phys]
    const int src = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int N = lb * k;
    const long long base = (long long)src * N;
    for (int i = threadIdx.x; i < W * (R + E_phys); i += blockDim.x) smem[i] = 0;
    __syncthreads();

    const int rounds = (N + 31) / 32;
    const int rpw = (rounds + W - 1) / W;
    const int r0 = w * rpw, r1 = min(rounds, r0 + rpw);
    const unsigned lt = (1u << lane) - 1u;

    for (int r = r0; r < r1; ++r) {
        int i = r * 32 + lane;
        const bool valid = i < N;
        int p = valid ? phys_idx[base + i] : -1;
        const bool ok = valid && p >= 0 && p < E_phys;  // caller data: keep the id in range
        if (valid && !ok) post_status(err, MOE_ERR_INDEX);
        p = ok ? p : -1;
        int dst = ok ? p / epr : -1;
        unsigned pd = __match_any_sync(0xffffffffu, dst);
        unsigned pe = __match_any_sync(0xffffffffu, p);
        if (ok && (pd & lt) == 0) cntD[w * R + dst] += __popc(pd);
        if (ok && (pe & lt) == 0) cntE[w * E_phys + p] += __popc(pe);
        __syncwarp();
    }
    __syncthreads();
    for (int b = threadIdx.x; b < R; b += blockDim.x) {
        int run = 0;
        for (int ww = 0; ww < W; ++ww) {
            int c = cntD[ww * R + b];
            cntD[ww * R + b] = run;
            run += c;
        }
        totD[b] = run;
    }
    for (int b = threadIdx.x; b < E_phys; b += blockDim.x) {
        int run = 0;
        for (int ww = 0; ww < W; ++ww) {
            int c = cntE[ww * E_phys + b];
            cntE[ww * E_phys + b] = run;
            run += c;
        }
        totE[b] = run;
    }
    __syncthreads();
    for (int r = r0; r < r1; ++r) {
        int i = r * 32 + lane;
        const bool valid = i < N;
        int p = valid ? phys_idx[base + i] : -1;
        const bool ok = valid && p >= 0 && p < E_phys;
        p = ok ? p : -1;
        int dst = ok ? p / epr : -1;
        unsigned pd = __match_any_sync(0xffffffffu, dst);
        unsigned pe = __match_any_sync(0xffffffffu, p);
        int sl = -1, er = 0;
        if (ok) {
            sl = cntD[w * R + dst] + __popc(pd & lt);
            er = cntE[w * E_phys + p] + __popc(pe & lt);
            if (sl >= mt) {  // the pair's static area is full: drop the message
                post_status(err, MOE_ERR_CAPACITY);
                sl = -1;
            }
        }
        __syncwarp();
        if (ok && (pd & lt) == 0) cntD[w * R + dst] += __popc(pd);
        if (ok && (pe & lt) == 0) cntE[w * E_phys + p] += __popc(pe);
        __syncwarp();
        if (valid) {
            slot_local[base + i] = sl;
            erank[base + i] = er;
        }
    }
    // messages actually placed in each pair's area (at most max_tokens)
    for (int b = threadIdx.x; b < R; b += blockDim.x) rank_counts[(long long)b * S + src] = min(totD[b], mt);
    for (int b = threadIdx.x; b < E_phys; b += blockDim.x) hist[(long long)src * E_phys + b] = totE[b];
}

__global__ void __launch_bounds__(1024)
layout_expert_kernel(int S, int E_phys, const int32_t* __restrict__ hist,
                     int32_t* __restrict__ src_base, int32_t* __restrict__ expert_offsets) {
    __shared__ int s_warp[32];
    const int p = threadIdx.x;
    int run = 0;
    if (p < E_phys) {
        for (int s = 0; s < S; ++s) {
            int c = hist[(long long)s * E_phys + p];
            src_base[(long long)s * E_phys + p] = run;
            run += c;
        }
    }
    // exclusive scan of run over p (block of 1024 threads)
    const int lane = p & 31, w = p >> 5;
    int v = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) s_warp[w] = v;
    __syncthreads();
    if (w == 0) {
        int x = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += o;
        }
        s_warp[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    int incl = v + (w > 0 ? s_warp[w - 1] : 0);
    if (p < E_phys) expert_offsets[p] = incl - run;
    if (p == E_phys - 1) expert_offsets[E_phys] = incl;
}

__device__ __forceinline__ void bulk_store_s2g(void* gdst, const void* ssrc, unsigned bytes) {
    unsigned saddr = static_cast<unsigned>(__cvta_generic_to_shared(ssrc));
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst),
                 "r"(saddr), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ unsigned pack4(int q0, int q1, int q2, int q3) {
    return (unsigned)(q0 & 0xff) | ((unsigned)(q1 & 0xff) << 8) | ((unsigned)(q2 & 0xff) << 16) |
           ((unsigned)(q3 & 0xff) << 24);
}

constexpr int kScatterThreads = 128;
constexpr int kLoadUnroll = 8;
constexpr int kMaxRoutes = 32;  // k <= 32 (checked by every entry point)

// Dispatch modes of the scatter kernel:
//   kDirect: quantise token t and write its k messages into the owners'
//            static areas (FusedDispatch);
//   kHop1:   quantise token t and write it once, with its k physical expert
//            ids, into its trampoline's area (the first hop of the
//            trampoline forward, "xDeepServe", P045);
//   kHop2:   read token t back from the trampoline area and write its k
//            messages exactly as kDirect does (the second hop).
enum { kDirect = 0, kHop1 = 1, kHop2 = 2 };

template <int MODE>
__global__ void __launch_bounds__(kScatterThreads)
scatter_kernel(int H, int k, int lb, int epr, int S, int mt, int E_phys, int int8_msgs,
               long long drow, const uint16_t* __restrict__ x,
               const int32_t* __restrict__ phys_idx, const int32_t* __restrict__ slot_local,
               const int32_t* __restrict__ erank, const int32_t* __restrict__ src_base,
               const int32_t* __restrict__ expert_offsets, char* __restrict__ dbuf,
               moe_dispatch_meta* __restrict__ meta, int32_t* __restrict__ expert_rows,
               char* __restrict__ trows, moe_dispatch_meta* __restrict__ tmeta,
               int32_t* __restrict__ troutes, __half* __restrict__ a16, float* __restrict__ s_row) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint4* srow = reinterpret_cast<uint4*>(sm);                 // bf16 row, 2H bytes
    uint2* scode = reinterpret_cast<uint2*>(sm + 2 * (size_t)H);  // H codes
    __shared__ float s_red[kScatterThreads / 32];
    __shared__ float s_scale;
    __shared__ long long s_slot[kMaxRoutes];  // kDirect: message slot of each route
    __shared__ int s_erow[kMaxRoutes];        // kDirect with a16: expert row of each route

    const int t = blockIdx.x;
    const int src = t / lb, bs = t - src * lb;
    const int nch = H / 8;  // 16-byte chunks of 8 bf16
    const long long tk = (long long)t * k;
    // kDirect, kHop2: the route threads look up their message slots and expert
    // row positions first, so that these dependent loads overlap the row's
    // loads.  my_slot < 0: no message is written (a physical id outside
    // [0, E_phys), or a full static area); for a full area the expert's row
    // list still gets an entry, pointed at the pair's last slot (written by
    // another message), so that every entry names a written slot.
    long long my_slot = -1, my_fill = -1;
    int my_erow = -1;
    if (MODE != kHop1 && threadIdx.x >= 32 && threadIdx.x < 32 + k) {
        const int j = threadIdx.x - 32;
        const int p = MODE == kHop2 ? troutes[tk + j] : phys_idx[tk + j];
        if (p >= 0 && p < E_phys) {
            const int sl = slot_local[tk + j];
            const long long pair = ((long long)(p / epr) * S + src) * mt;
            my_erow = expert_offsets[p] + src_base[(long long)src * E_phys + p] + erank[tk + j];
            my_slot = sl >= 0 ? pair + sl : -1;
            my_fill = pair + mt - 1;
        }
        s_slot[j] = my_slot;
        s_erow[j] = my_erow;
    }
    if constexpr (MODE == kHop2) {
        // the token as the trampoline holds it: the message row, its scale and routes
        const uint4* tr = reinterpret_cast<const uint4*>(trows + (long long)t * drow);
        uint4* dstm = reinterpret_cast<uint4*>(sm);
        for (int c = threadIdx.x; c < (int)(drow / 16); c += kScatterThreads) dstm[c] = tr[c];
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncthreads();
        const float scale = tmeta[t].scale;
        if (threadIdx.x == 0) {
            for (int j = 0; j < k; ++j)
                if (s_slot[j] >= 0) bulk_store_s2g(dbuf + s_slot[j] * drow, sm, (unsigned)drow);
            asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
        }
        if (threadIdx.x >= 32 && threadIdx.x < 32 + k) {
            if (my_slot >= 0) {
                moe_dispatch_meta m;
                m.scale = scale;
                m.src_rank = src;
                m.batch_slot = bs;
                m.route_slot = threadIdx.x - 32;
                meta[my_slot] = m;
                expert_rows[my_erow] = (int32_t)my_slot;
            } else if (my_erow >= 0) {
                expert_rows[my_erow] = (int32_t)my_fill;
            }
        }
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
        return;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(x + (long long)t * H);
    float amax = 0.f;
    // up to kLoadUnroll 16-byte loads of the row in flight per thread
    for (int c0 = threadIdx.x; c0 < nch; c0 += kLoadUnroll * kScatterThreads) {
        uint4 v[kLoadUnroll];
#pragma unroll
        for (int u = 0; u < kLoadUnroll; ++u) {
            const int c = c0 + u * kScatterThreads;
            if (c < nch) v[u] = __ldg(xr + c);
        }
#pragma unroll
        for (int u = 0; u < kLoadUnroll; ++u) {
            const int c = c0 + u * kScatterThreads;
            if (c < nch) {
                srow[c] = v[u];
                if (int8_msgs) {
                    amax = fmaxf(amax, fabsf(bf16_lo(v[u].x)));
                    amax = fmaxf(amax, fabsf(bf16_hi(v[u].x)));
                    amax = fmaxf(amax, fabsf(bf16_lo(v[u].y)));
                    amax = fmaxf(amax, fabsf(bf16_hi(v[u].y)));
                    amax = fmaxf(amax, fabsf(bf16_lo(v[u].z)));
                    amax = fmaxf(amax, fabsf(bf16_hi(v[u].z)));
                    amax = fmaxf(amax, fabsf(bf16_lo(v[u].w)));
                    amax = fmaxf(amax, fabsf(bf16_hi(v[u].w)));
                }
            }
        }
    }
    const unsigned char* src_row = sm;
    float scale = 0.f;
    if (int8_msgs) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
        __syncthreads();
        if (threadIdx.x == 0) {
            float a = s_red[0];
            for (int i = 1; i < kScatterThreads / 32; ++i) a = fmaxf(a, s_red[i]);
            s_scale = a == 0.f ? 0.f : __fdiv_rn(a, 127.0f);
        }
        __syncthreads();
        scale = s_scale;
        const float rscale = quant_rcp(scale);
        for (int c = threadIdx.x; c < nch; c += kScatterThreads) {
            uint4 v = srow[c];
            uint2 q;
            if (scale == 0.f) {
                q.x = 0u; q.y = 0u;
            } else {
                const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                                    bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
                int c8[8];
                quant_row_n<8>(x, scale, rscale, c8);
                q.x = pack4(c8[0], c8[1], c8[2], c8[3]);
                q.y = pack4(c8[4], c8[5], c8[6], c8[7]);
                if (MODE == kDirect && a16)  // the chunk's codes as fp16, over its bf16 values
                    srow[c] = make_uint4(codes_to_f16x2(c8[0], c8[1]), codes_to_f16x2(c8[2], c8[3]),
                                         codes_to_f16x2(c8[4], c8[5]), codes_to_f16x2(c8[6], c8[7]));
            }
            if (MODE == kDirect && a16 && scale == 0.f) srow[c] = make_uint4(0u, 0u, 0u, 0u);
            scode[c] = q;
        }
        src_row = reinterpret_cast<const unsigned char*>(scode);
    }
    // generic-proxy shared writes -> visible to the bulk-copy (async) proxy
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if constexpr (MODE == kHop1) {
        // one copy of the token, its scale and its routes to the trampoline
        if (threadIdx.x == 0) {
            bulk_store_s2g(trows + (long long)t * drow, src_row, (unsigned)drow);
            asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            moe_dispatch_meta m;
            m.scale = scale;
            m.src_rank = src;
            m.batch_slot = bs;
            m.route_slot = k;  // the k routes follow in troutes
            tmeta[t] = m;
        }
        if (threadIdx.x >= 32 && threadIdx.x < 32 + k) troutes[tk + threadIdx.x - 32] = phys_idx[tk + threadIdx.x - 32];
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
        return;
    }
    if (threadIdx.x == 0) {
        for (int j = 0; j < k; ++j)
            if (s_slot[j] >= 0) bulk_store_s2g(dbuf + s_slot[j] * drow, src_row, (unsigned)drow);
        // moe_layer: the expert FFN's input rows too (the expert-input assembly
        // of the tensor-core FFN, done here from the codes in shared memory)
        if (a16 && int8_msgs)
            for (int j = 0; j < k; ++j)
                if (s_erow[j] >= 0) bulk_store_s2g(a16 + (long long)s_erow[j] * H, sm, (unsigned)(2 * H));
        asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
    }
    if (threadIdx.x >= 32 && threadIdx.x < 32 + k) {
        if (a16 && int8_msgs && my_erow >= 0) s_row[my_erow] = scale;
        if (my_slot >= 0) {
            moe_dispatch_meta m;
            m.scale = scale;
            m.src_rank = src;
            m.batch_slot = bs;
            m.route_slot = threadIdx.x - 32;
            meta[my_slot] = m;
            expert_rows[my_erow] = (int32_t)my_slot;
        } else if (my_erow >= 0) {
            expert_rows[my_erow] = (int32_t)my_fill;
        }
    }
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

}  // namespace

namespace {

// The two layout kernels: per-(destination, source) slots, per-expert counts,
// offsets and the per-source bases of the expert row lists.
cudaError_t launch_layout(const Dims& d, const int32_t* phys_idx, int32_t* rank_counts,
                          int32_t* expert_offsets, void* ws, const WsLayout& wl, cudaStream_t st) {
    int32_t* slot_local = ws_ptr<int32_t>(ws, wl.slot_local);
    int32_t* erank = ws_ptr<int32_t>(ws, wl.erank);
    int32_t* hist = ws_ptr<int32_t>(ws, wl.hist);
    int32_t* src_base = ws_ptr<int32_t>(ws, wl.src_base);
    // warps per source: one per 32-message round, between 4 (the per-rank and
    // per-expert passes use every thread of the block) and kLayoutMaxWarps;
    // fewer if their per-warp counters would not fit in shared memory
    const long long rounds = ((long long)d.lb * d.k + 31) / 32;
    const size_t per_warp = sizeof(int) * (size_t)(d.R + d.E_phys);
    int W = (int)std::min<long long>(kLayoutMaxWarps, std::max<long long>(4, rounds));
    while (W > 1 && (size_t)(W + 1) * per_warp > 48 * 1024) --W;
    const size_t smem1 = (size_t)(W + 1) * per_warp;
    if (smem1 > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(layout_src_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem1);
        if (e != cudaSuccess) return e;
    }
    layout_src_kernel<<<d.S, W * 32, smem1, st>>>(d.lb, d.k, d.epr, d.R, d.E_phys, d.S, d.mt,
                                                  phys_idx, slot_local, erank, rank_counts, hist,
                                                  ws_ptr<int>(ws, 0));
    layout_expert_kernel<<<1, 1024, 0, st>>>(d.S, d.E_phys, hist, src_base, expert_offsets);
    count_launches(2);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_scatter(const Dims& d, const uint16_t* x, const int32_t* phys_idx, void* dbuf,
                           long long meta_off, int32_t* expert_offsets, int32_t* expert_rows,
                           void* ws, const WsLayout& wl, char* trows, moe_dispatch_meta* tmeta,
                           int32_t* troutes, cudaStream_t st, bool stage_rows = false) {
    size_t smem3 = (size_t)d.H * 2 + (d.dfmt == MOE_MSG_INT8 ? (size_t)d.H : 0);
    if (smem3 > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(scatter_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem3);
        if (e != cudaSuccess) return e;
    }
    scatter_kernel<MODE><<<d.T, kScatterThreads, smem3, st>>>(
        d.H, d.k, d.lb, d.epr, d.S, d.mt, d.E_phys, d.dfmt == MOE_MSG_INT8 ? 1 : 0, d.drow, x,
        phys_idx, ws_ptr<int32_t>(ws, wl.slot_local), ws_ptr<int32_t>(ws, wl.erank),
        ws_ptr<int32_t>(ws, wl.src_base), expert_offsets, static_cast<char*>(dbuf),
        reinterpret_cast<moe_dispatch_meta*>(static_cast<char*>(dbuf) + meta_off), expert_rows,
        trows, tmeta, troutes, stage_rows ? ws_ptr<__half>(ws, wl.a16) : nullptr,
        stage_rows ? ws_ptr<float>(ws, wl.s_row) : nullptr);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const Dims& d, const uint16_t* x, const int32_t* phys_idx,
                            void* dbuf, long long meta_off, int32_t* rank_counts,
                            int32_t* expert_offsets, int32_t* expert_rows, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear, bool stage_rows) {
    cudaError_t e = clear ? clear_status(ws, st) : cudaSuccess;
    if (e != cudaSuccess) return e;
    e = launch_layout(d, phys_idx, rank_counts, expert_offsets, ws, wl, st);
    if (e != cudaSuccess) return e;
    return launch_scatter<kDirect>(d, x, phys_idx, dbuf, meta_off, expert_offsets, expert_rows, ws,
                                   wl, nullptr, nullptr, nullptr, st,
                                   stage_rows && wl.tc && d.dfmt == MOE_MSG_INT8);
}

TrampolineLayout trampoline_layout(const Dims& d) {
    TrampolineLayout t;
    t.rows = 0;
    t.meta = align_up((long long)d.T * d.drow, 256);
    t.routes = align_up(t.meta + 16LL * d.T, 256);
    t.total = align_up(t.routes + 4LL * d.T * d.k, 256);
    return t;
}

cudaError_t launch_dispatch_trampoline(const Dims& d, const uint16_t* x, const int32_t* phys_idx,
                                       void* tbuf, void* dbuf, long long meta_off,
                                       int32_t* rank_counts, int32_t* expert_offsets,
                                       int32_t* expert_rows, void* ws, const WsLayout& wl,
                                       cudaStream_t st) {
    const TrampolineLayout tl = trampoline_layout(d);
    cudaError_t e0 = clear_status(ws, st);
    if (e0 != cudaSuccess) return e0;
    char* tb = static_cast<char*>(tbuf);
    char* trows = tb + tl.rows;
    moe_dispatch_meta* tmeta = reinterpret_cast<moe_dispatch_meta*>(tb + tl.meta);
    int32_t* troutes = reinterpret_cast<int32_t*>(tb + tl.routes);
    cudaError_t e = launch_scatter<kHop1>(d, x, phys_idx, dbuf, meta_off, expert_offsets,
                                          expert_rows, ws, wl, trows, tmeta, troutes, st);
    if (e != cudaSuccess) return e;
    if ((e = launch_layout(d, phys_idx, rank_counts, expert_offsets, ws, wl, st)) != cudaSuccess)
        return e;
    return launch_scatter<kHop2>(d, nullptr, nullptr, dbuf, meta_off, expert_offsets, expert_rows,
                                 ws, wl, trows, tmeta, troutes, st);
}

}  // namespace moe
