// ffn_gemv.cu -- the expert FFN for decode batches with a few routed rows
// per expert: the grouped GEMMs as streamed matrix-vector products on the
// CUDA cores.
//
// "xDeepServe on CloudMatrix384", section "DeepSeek INT8 量化": P085 (token-wise
// activation scale s_i, channel-wise weight scale s^w_j, y_ij ~ s_i s^w_j
// sum_k q(x_ik) q(w_jk)), P088 (gate_proj and up_proj computed together).
// "CloudMatrix384 LLM Serving", section "EP320：token 去找专家"
// (run_local_experts).
//
// With one to a few tokens per expert (a decode step: T = 96, k = 8 over 256
// experts routes about 3 rows to each), the expert FFN reads every touched
// weight once and does almost no arithmetic per weight byte.  The tensor-core
// GEMM still pays its whole pipeline per 64-K stage for those few tokens; here
// each warp streams 8 weight rows with coalesced 16-byte loads and forms the
// dot products with the (at most 8) token rows of its expert, held in shared
// memory, by dp4a: four int8 products summed into int32, exact.  The outputs
// are those of the tensor-core path, bit for bit: g and u in f32 (gate/up;
// SwiGLU follows in the requantisation kernel), y in f32 with its per-row
// |y| maximum (down); requant_rows and retquant_rows take it from there.
//
// Block (256 threads, 8 warps) = one expert and 32 gate/up channel pairs
// (gate/up), or one expert and 4 groups of 64 output channels (down: its
// rows are only I = 2048 bytes long, so a block takes 256 of them to spread
// the staging of its token rows over 512 KB of weights).  Warp w takes 8
// weight rows at a time: gate channels 4w..4w+3 of the block and the matching
// up channels, or output channels 8w..8w+7 of each down group.  A lane reads 16 bytes of each row
// per 512-byte step of K.  Experts with more than 8 rows are done 8 at a time.
// After the K loop the warp's 64 partial sums (8 rows x 8 tokens) are reduced
// over the lanes by a reduce-scatter of shuffles (62 exchanges), which leaves
// lane L with the finished sums of row L / 4 and tokens 2(L % 4), 2(L % 4)+1.
#include <algorithm>
#include <climits>
#include <cuda_fp16.h>

#include "device_math.cuh"
#include "internal.cuh"

namespace moe {
namespace gv {

constexpr int NT = 8;        // token rows per pass
constexpr int ROWS = 8;      // weight rows per warp
constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;
constexpr int KSTEP = 512;   // K bytes per warp step (32 lanes x 16 bytes)
constexpr int DOWN_GROUPS = 4;  // 64-channel groups per down block (256 channels)

enum { GATE_UP = 0, DOWN = 1 };

struct Params {
    const int32_t* offsets;       // [E+1] expert row offsets
    const int32_t* p2w;           // nullable: weight set of each physical expert
    const int8_t* w;              // weights: [set][2I][H] (gate rows, then up rows) or [set][H][I]
    const float* s_ch;            // channel scales [set][2I] or [set][H]
    int K;                        // H (gate/up) or I (down), multiple of KSTEP
    int nout;                     // I (gate/up) or H (down)
    // activations: gate/up reads int8 dispatch codes through expert_rows,
    // down reads the fp16 codes of h
    const int32_t* expert_rows;
    const int8_t* dbuf;
    long long drow;
    const moe_dispatch_meta* meta;
    const __half* hq16;
    const float* s_h;             // down: per-row scale of h
    float* out;                   // g and u [M][2I] (gate/up) or y [M][H] (down)
    unsigned* rowmax;             // down: [M] |y| maximum (float bits)
    long long M;                  // routed rows (rows of out)
    long long nslots;             // dispatch slots (rows of dbuf)
    int n_sets;                   // weight sets
    const int32_t* list;          // null: block row y takes expert y; else the experts list[1..list[0]]
    int* err;                     // workspace status word
};

// 16 bytes of a weight row that is read once: no L1 allocation.
__device__ __forceinline__ int4 ld_stream(const int8_t* p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Reduce-scatter of 64 values over the 32 lanes of a warp: afterwards a[0]
// and a[1] of lane L hold the warp sums of values 2L and 2L + 1.
__device__ __forceinline__ void reduce_scatter64(int (&a)[ROWS * NT], int lane) {
#pragma unroll
    for (int d = 16, n = 32; d >= 1; d >>= 1, n >>= 1) {
        const bool hi = lane & d;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (i < n) {
                const int send = hi ? a[i] : a[i + n];
                const int keep = hi ? a[i + n] : a[i];
                a[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
            }
        }
    }
}

// One expert's share of the block: output channels blockIdx.x of expert e.
// xs [NT][K] holds a pass's token rows, s_tok their scales.
template <int KIND>
__device__ __forceinline__ void gemv_expert(const Params& P, int e, int8_t* xs, float* s_tok) {
    const int r_begin = P.offsets[e], r_end = P.offsets[e + 1];
    if (r_begin == r_end) return;
    const int set = P.p2w ? P.p2w[e] : e;
    // offsets and weight sets are caller data: an expert whose rows or
    // weight set fall outside the buffers is skipped
    if (r_begin < 0 || r_end < r_begin || r_end > P.M || set < 0 || set >= P.n_sets) {
        if (threadIdx.x == 0) post_status(P.err, MOE_ERR_INDEX);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = P.K;
    // this warp's weight rows
    const int8_t* wrow[ROWS];
    int ch0;  // first output channel of the warp
    if constexpr (KIND == GATE_UP) {
        ch0 = blockIdx.x * 32 + warp * 4;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const long long wr = (long long)set * 2 * P.nout + (r < 4 ? 0 : P.nout) + ch0 + (r & 3);
            wrow[r] = P.w + wr * K + lane * 16;
        }
    } else {
        ch0 = blockIdx.x * 64 * DOWN_GROUPS + warp * 8;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) wrow[r] = P.w + ((long long)set * P.nout + ch0 + r) * K + lane * 16;
    }

    for (int t0 = r_begin; t0 < r_end; t0 += NT) {
        const int n = min(NT, r_end - t0);
        __syncthreads();  // the previous pass has finished with xs
        // stage the pass's token rows as int8
        if constexpr (KIND == GATE_UP) {
            const int nvec = K / 16;
            // a row-list entry outside the dispatch buffer reads as a zero row
            for (int i = threadIdx.x; i < n * nvec; i += THREADS) {
                const int t = i / nvec, c = i - t * nvec;
                const long long slot = P.expert_rows[t0 + t];
                int4 v = make_int4(0, 0, 0, 0);
                if (slot >= 0 && slot < P.nslots)
                    v = __ldg(reinterpret_cast<const int4*>(P.dbuf + slot * P.drow) + c);
                reinterpret_cast<int4*>(xs + t * K)[c] = v;
            }
            if (threadIdx.x < n) {
                const long long slot = P.expert_rows[t0 + threadIdx.x];
                const bool ok = slot >= 0 && slot < P.nslots;
                if (!ok) post_status(P.err, MOE_ERR_INDEX);
                s_tok[threadIdx.x] = ok ? P.meta[slot].scale : 0.f;
            }
        } else {
            const int nvec = K / 8;  // 8 fp16 codes -> 8 int8
            for (int i = threadIdx.x; i < n * nvec; i += THREADS) {
                const int t = i / nvec, c = i - t * nvec;
                const uint4 h = __ldg(reinterpret_cast<const uint4*>(P.hq16 + (long long)(t0 + t) * K) + c);
                const __half2* hh = reinterpret_cast<const __half2*>(&h);
                uint32_t q[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float2 a = __half22float2(hh[2 * u]), b = __half22float2(hh[2 * u + 1]);
                    q[u] = (uint32_t)((int)a.x & 0xff) | ((uint32_t)((int)a.y & 0xff) << 8) |
                           ((uint32_t)((int)b.x & 0xff) << 16) | ((uint32_t)((int)b.y & 0xff) << 24);
                }
                reinterpret_cast<uint2*>(xs + t * K)[c] = make_uint2(q[0], q[1]);
            }
            if (threadIdx.x < n) s_tok[threadIdx.x] = P.s_h[t0 + threadIdx.x];
        }
        __syncthreads();

        for (int g = 0; g < (KIND == DOWN ? DOWN_GROUPS : 1); ++g) {
            const long long goff = (long long)g * 64 * K;  // down: rows of group g
            int acc[ROWS * NT];
#pragma unroll
            for (int i = 0; i < ROWS * NT; ++i) acc[i] = 0;
#pragma unroll 2
            for (int k = 0; k < K; k += KSTEP) {
                int4 wv[ROWS];
#pragma unroll
                for (int r = 0; r < ROWS; ++r) wv[r] = ld_stream(wrow[r] + goff + k);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t < n) {
                        const int4 x = *reinterpret_cast<const int4*>(xs + t * K + k + lane * 16);
#pragma unroll
                        for (int r = 0; r < ROWS; ++r) {
                            int& s = acc[r * NT + t];
                            s = __dp4a(wv[r].x, x.x, s);
                            s = __dp4a(wv[r].y, x.y, s);
                            s = __dp4a(wv[r].z, x.z, s);
                            s = __dp4a(wv[r].w, x.w, s);
                        }
                    }
                }
            }
            reduce_scatter64(acc, lane);
            // lane L: row L >> 2, tokens tl and tl + 1
            const int row = lane >> 2, tl = 2 * (lane & 3);
            if constexpr (KIND == GATE_UP) {
                // lanes 0..15 hold gate rows, lanes 16..31 the up rows of the same
                // channels and tokens: each writes its scaled projection, g to
                // column c and u to column I + c of the token's [2I] row
                const int col = (lane < 16 ? 0 : P.nout) + ch0 + (row & 3);
                const float sc = P.s_ch[(long long)set * 2 * P.nout + col];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = tl + u;
                    if (t < n)
                        P.out[(long long)(t0 + t) * 2 * P.nout + col] =
                            __fmul_rn(__fmul_rn(__int2float_rn(acc[u]), s_tok[t]), sc);
                }
            } else {
                const int c = ch0 + g * 64 + row;
                const float sd = P.s_ch[(long long)set * P.nout + c];
                float mx[2] = {0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = tl + u;
                    if (t < n) {
                        const float y = __fmul_rn(__fmul_rn(__int2float_rn(acc[u]), s_tok[t]), sd);
                        P.out[(long long)(t0 + t) * P.nout + c] = y;
                        mx[u] = fabsf(y);
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float m = mx[u];
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    if (row == 0 && tl + u < n) atomicMax(&P.rowmax[t0 + tl + u], __float_as_uint(m));
                }
            }
        }
    }
}

// Every pass of gemv_expert starts with a block barrier before it stages
// token rows, so consecutive experts of one block never overlap in xs.
template <int KIND>
__global__ void __launch_bounds__(THREADS, 2) gemv_kernel(const Params P) {
    extern __shared__ __align__(16) int8_t xs[];  // [NT][K] token rows of the current expert
    __shared__ float s_tok[NT];                   // their scales
    if (P.list == nullptr) {
        gemv_expert<KIND>(P, blockIdx.y, xs, s_tok);
        return;
    }
    const int n = P.list[0];
    for (int i = blockIdx.y; i < n; i += gridDim.y) gemv_expert<KIND>(P, P.list[1 + i], xs, s_tok);
}

// Blocks of a list-mode launch (the narrow experts beside the tensor-core
// GEMMs, whose number only the device knows): at c2_decode_zipf (101 narrow
// experts) 1024 blocks, each looping over about six experts, streamed the
// weights at 5.66 TB/s; 4096, most blocks taking one expert, at 6.21 TB/s
// (2048: 6.13, 8192 and 16384: 6.20).
constexpr int kListBlocks = 4096;

// Grid: nblocks_x channel blocks times E experts (no list), or times enough
// block rows to cover kListBlocks blocks (list: the rows stride over the
// listed experts; rows beyond the list's length end at once).
template <int KIND>
cudaError_t launch(const Params& P, int E, int nblocks_x, cudaStream_t st) {
    if (P.list != nullptr) E = std::max(1, std::min(E, (kListBlocks + nblocks_x - 1) / nblocks_x));
    const size_t smem = (size_t)NT * P.K;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<KIND><<<dim3((unsigned)nblocks_x, (unsigned)E), THREADS, smem, st>>>(P);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace gv

bool gemv_kernels_fit(const Dims& d) {
    return d.cfmt == MOE_MSG_INT8 && d.H % gv::KSTEP == 0 && d.I % gv::KSTEP == 0 &&
           (size_t)gv::NT * d.H <= 200 * 1024;
}

bool ffn_gemv_fits(const Dims& d) {
    const long long M = (long long)d.T * d.k;
    return gemv_kernels_fit(d) && M <= (long long)kGemvRowsPerExpert * d.E_phys;
}

cudaError_t launch_gemv_gate_up(const Dims& d, const void* dbuf, const moe_dispatch_meta* meta,
                                const int32_t* expert_offsets, const int32_t* expert_rows,
                                const moe_expert_weights& w, float* gubuf, int* err,
                                const int32_t* list, int prof_slot, cudaStream_t st) {
    gv::Params P = {};
    P.offsets = expert_offsets; P.p2w = w.phys_to_weight; P.w = w.w_gate_up; P.s_ch = w.s_gate_up;
    P.K = d.H; P.nout = d.I;
    P.expert_rows = expert_rows; P.dbuf = static_cast<const int8_t*>(dbuf); P.drow = d.drow; P.meta = meta;
    P.out = gubuf;
    P.M = (long long)d.T * d.k; P.nslots = d.nslots; P.n_sets = w.n_sets; P.list = list; P.err = err;
    if (cudaEvent_t ev = prof_event(prof_slot, 0)) cudaEventRecord(ev, st);
    cudaError_t e = gv::launch<gv::GATE_UP>(P, d.E_phys, d.I / 32, st);
    if (cudaEvent_t ev = prof_event(prof_slot, 1)) cudaEventRecord(ev, st);
    return e;
}

cudaError_t launch_gemv_down(const Dims& d, const int32_t* expert_offsets, const moe_expert_weights& w,
                             const void* hq16, const float* sh, float* ybuf, unsigned* ymax, int* err,
                             const int32_t* list, int prof_slot, cudaStream_t st) {
    gv::Params P = {};
    P.offsets = expert_offsets; P.p2w = w.phys_to_weight; P.w = w.w_down; P.s_ch = w.s_down;
    P.K = d.I; P.nout = d.H;
    P.hq16 = static_cast<const __half*>(hq16); P.s_h = sh;
    P.out = ybuf; P.rowmax = ymax;
    P.M = (long long)d.T * d.k; P.nslots = d.nslots; P.n_sets = w.n_sets; P.list = list; P.err = err;
    if (cudaEvent_t ev = prof_event(prof_slot, 0)) cudaEventRecord(ev, st);
    cudaError_t e = gv::launch<gv::DOWN>(P, d.E_phys, d.H / (64 * gv::DOWN_GROUPS), st);
    if (cudaEvent_t ev = prof_event(prof_slot, 1)) cudaEventRecord(ev, st);
    return e;
}

cudaError_t launch_ffn_gemv(const Dims& d, const void* dbuf, long long meta_off,
                            const int32_t* expert_offsets, const int32_t* expert_rows,
                            const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear) {
    const long long M = (long long)d.T * d.k;
    const moe_dispatch_meta* meta =
        reinterpret_cast<const moe_dispatch_meta*>(static_cast<const char*>(dbuf) + meta_off);
    int* err = ws_ptr<int>(ws, 0);
    float* sh = ws_ptr<float>(ws, wl.sh);
    float* gubuf = ws_ptr<float>(ws, wl.gubuf);
    unsigned* ymax = ws_ptr<unsigned>(ws, wl.rowmax);
    void* hq16 = ws_ptr<void>(ws, wl.hq16);
    float* ybuf = ws_ptr<float>(ws, wl.ybuf);
    cudaError_t e;
    if (clear && (e = clear_status(ws, st)) != cudaSuccess) return e;
    if ((e = launch_gemv_gate_up(d, dbuf, meta, expert_offsets, expert_rows, w, gubuf, err, nullptr, 0,
                                 st)) != cudaSuccess)
        return e;
    if ((e = launch_requant_rows(d.I, M, gubuf, hq16, sh, ymax, st)) != cudaSuccess) return e;
    if ((e = launch_gemv_down(d, expert_offsets, w, hq16, sh, ybuf, ymax, err, nullptr, 1, st)) != cudaSuccess)
        return e;
    return launch_retquant_rows(d, M, ybuf, ymax, expert_rows, meta, static_cast<unsigned char*>(cbuf),
                                reinterpret_cast<float*>(static_cast<unsigned char*>(cbuf) + scale_off), err,
                                st);
}

}  // namespace moe
