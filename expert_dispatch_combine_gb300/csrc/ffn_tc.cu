// ffn_tc.cu -- grouped exact-INT8 expert GEMM on the 5th-generation tensor
// cores (tcgen05), plus the expert-FFN steps around it.
//
// "xDeepServe on CloudMatrix384", section "DeepSeek INT8 量化": P085 (token-wise
// activation scale s_i, channel-wise weight scale s^w_j, y_ij ~ s_i s^w_j
// sum_k q(x_ik) q(w_jk)), P088 (gate_proj and up_proj fused in one kernel),
// P089 (expert outputs quantised to INT8 for the return trip).
// "CloudMatrix384 LLM Serving", section "EP320：token 去找专家"
// (assemble_expert_inputs, run_local_experts, remote_write_combine).
//
// sm_103a has no integer tcgen05.mma, so the int8 contraction runs on
// kind::f16: every int8 value is exact in fp16, every product (|p| <= 16129)
// is exact in fp32, and the fp32 accumulator is drained to int32 every 1024
// K (1024 * 16129 < 2^24, so every partial sum is an exact integer).  The
// int32 results equal the integer matrix product bit for bit.
//
// GEMM structure (one CTA per SM, persistent over tiles):
//   D^T[channel][token] = W[channel][:] . X[token][:]
//   A operand = weights (128 channel rows): TMA loads int8 tiles into shared
//     memory; a converter warpgroup turns them into fp16 and stores them in
//     tensor memory (A-from-TMEM form of tcgen05.mma), so the converted
//     weights cost no shared-memory bandwidth;
//   B operand = activations (up to 128 tokens, fp16, K-major, 128B swizzle),
//     TMA-loaded into shared memory;
//   D = two 128x128 fp32 accumulators in TMEM (double-buffered across the
//     1024-K chunks) plus 128 columns of int32 running sums.
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2-5 converter / chunk drain / epilogue (one TMEM lane quarter each).
// The MMA N is the tile's token count rounded up to 16, so small experts do
// not pay for padding.  Every mbarrier wait is bounded (2 s): on a timeout
// the kernel records MOE_ERR_TIMEOUT in the workspace status word, waits
// briefly for its own copies in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_math.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BN = 128;                          // tokens per tile
constexpr int BK = 64;                           // K per stage
constexpr int NS = 8;                            // shared-memory stages
constexpr int NA = 4;                            // TMEM A slots
constexpr int CK = 16;                           // stages per exact chunk (1024 K)
constexpr int B_BYTES = BN * BK * 2;             // fp16 activations per stage
constexpr int A_BYTES = 128 * BK;                // int8 weights per stage
constexpr int STAGE_BYTES = B_BYTES + A_BYTES;   // 24 KB
constexpr int XLD = 33;                          // exchange row pitch (floats)
constexpr int XCH_BYTES = 128 * XLD * 4;
constexpr int NBARS = 2 * NS + 2 * NA + 4 + 2;
constexpr uint32_t TM_ACC = 0, TM_SUM = 256, TM_A = 384, TM_COLS = 512;
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = NS * STAGE_BYTES + XCH_BYTES + NBARS * 8 + 16 + 1024;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 20000000ull;

enum { EPI_I32 = 0, EPI_SWIGLU = 1, EPI_DOWN_F32 = 2, EPI_DOWN_BF16 = 3 };

struct Params {
    int G;
    const int32_t* offsets;      // [G+1] token rows per group
    const int32_t* tile_prefix;  // [G+1] token tiles per group
    const int32_t* g2s;          // nullable: weight set of each group
    int K;                       // reduction length, multiple of 64
    int rows_per_set;            // weight rows per set
    int nout;                    // output channels (h channels for SwiGLU)
    int mb_count;                // channel blocks per token tile
    int box1_off;                // row offset of the second 64-row weight box
    const float* s_row;          // per token-row scale
    const float* s_ch;           // per-channel weight scales [set][rows_per_set]
    int32_t* c_i32;              // EPI_I32: [M][nout]
    float* out_f32;              // EPI_SWIGLU: h [M][nout]; EPI_DOWN_F32: y [M][nout]
    unsigned* rowmax;            // per token-row absmax (float bits)
    const int32_t* expert_rows;  // EPI_DOWN_BF16: row -> dispatch slot
    const moe_dispatch_meta* meta;
    unsigned char* cbuf;
    long long crow;
    int k, lb;
    int* err;
};

struct TileInfo {
    int p, set, r0, nvalid, nmma, mb;
};

__device__ __forceinline__ TileInfo decode(const Params& P, int tile) {
    TileInfo t;
    const int nt = tile / P.mb_count;
    t.mb = tile - nt * P.mb_count;
    t.p = find_group(P.tile_prefix, P.G, nt);
    t.r0 = P.offsets[t.p] + (nt - P.tile_prefix[t.p]) * BN;
    t.nvalid = min(BN, P.offsets[t.p + 1] - t.r0);
    t.nmma = (t.nvalid + 15) & ~15;
    t.set = P.g2s ? P.g2s[t.p] : t.p;
    return t;
}

// Warp-uniform bounded wait: every lane waits (each acquires the phase), and
// the warp goes on only if all lanes saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
    const bool ok = ptx::mbar_wait(bar, parity, err, WAIT_NS, MOE_ERR_TIMEOUT);
    return __all_sync(0xffffffffu, ok);
}

// Bounded barrier of the four converter warps (an mbarrier with count 4
// instead of bar.sync, so that a warp that gave up cannot hang the others).
struct WgBarrier {
    uint32_t addr;
    uint32_t phase;
    __device__ __forceinline__ bool sync(int lane, int* err) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(addr);
        const bool ok = warp_wait(addr, phase & 1, err);
        ++phase;
        return ok;
    }
};

// Wait without regard to the error word, with a short limit (used only to
// let copies already in flight land before the CTA exits).
__device__ __forceinline__ void mbar_wait_quiet(uint32_t bar, uint32_t parity, uint64_t limit) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try(bar, parity))
        if (ptx::globaltimer() - t0 > limit) break;
}

// Epilogue for one 32-token slice of a finished tile.  `row` is this
// thread's TMEM lane (weight channel within the tile), iv[j] the exact int32
// result for token j0 + j.
template <int EPI>
__device__ __forceinline__ bool epilogue_slice(const Params& P, const TileInfo& ti, int row,
                                               int j0, const int (&iv)[32], float* xch,
                                               WgBarrier& wg, int lane) {
    if constexpr (EPI == EPI_I32) {
        const int ch = ti.mb * 128 + row;
        if (ch < P.nout) {
#pragma unroll 4
            for (int j = 0; j < 32; ++j)
                if (j0 + j < ti.nvalid) P.c_i32[(long long)(ti.r0 + j0 + j) * P.nout + ch] = iv[j];
        }
    } else if constexpr (EPI == EPI_SWIGLU) {
        // rows 0..63: gate of channel i, rows 64..127: up of channel i
        const int i = ti.mb * 64 + (row & 63);
        const float* sc = P.s_ch + (long long)ti.set * P.rows_per_set;
        if (row >= 64) {
            const float su = sc[P.nout + i];
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const float st = (j0 + j < ti.nvalid) ? P.s_row[ti.r0 + j0 + j] : 0.f;
                xch[(row - 64) * XLD + j] = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), st), su);
            }
        }
        if (!wg.sync(lane, P.err)) return false;
        if (row < 64) {
            const float sg = sc[i];
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const bool ok = j0 + j < ti.nvalid;
                const float st = ok ? P.s_row[ti.r0 + j0 + j] : 0.f;
                const float g = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), st), sg);
                const float h = __fmul_rn(silu_spec(g), xch[row * XLD + j]);
                if (ok) P.out_f32[(long long)(ti.r0 + j0 + j) * P.nout + i] = h;
                xch[row * XLD + j] = ok ? fabsf(h) : 0.f;
            }
        }
        if (!wg.sync(lane, P.err)) return false;
        if (row < 32 && j0 + row < ti.nvalid) {
            float m = 0.f;
            for (int L = 0; L < 64; ++L) m = fmaxf(m, xch[L * XLD + row]);
            atomicMax(&P.rowmax[ti.r0 + j0 + row], __float_as_uint(m));
        }
        if (!wg.sync(lane, P.err)) return false;
    } else {
        const int ch = ti.mb * 128 + row;
        const bool chok = ch < P.nout;
        const float sd = chok ? P.s_ch[(long long)ti.set * P.rows_per_set + ch] : 0.f;
        if constexpr (EPI == EPI_DOWN_F32) {
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const bool ok = chok && (j0 + j < ti.nvalid);
                const float sr = (j0 + j < ti.nvalid) ? P.s_row[ti.r0 + j0 + j] : 0.f;
                const float y = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), sr), sd);
                if (ok) P.out_f32[(long long)(ti.r0 + j0 + j) * P.nout + ch] = y;
                xch[row * XLD + j] = ok ? fabsf(y) : 0.f;
            }
            if (!wg.sync(lane, P.err)) return false;
            if (row < 32 && j0 + row < ti.nvalid) {
                float m = 0.f;
                for (int L = 0; L < 128; ++L) m = fmaxf(m, xch[L * XLD + row]);
                atomicMax(&P.rowmax[ti.r0 + j0 + row], __float_as_uint(m));
            }
            if (!wg.sync(lane, P.err)) return false;
        } else {  // EPI_DOWN_BF16: the return message is bf16(y), written in place
#pragma unroll 2
            for (int j = 0; j < 32; ++j) {
                if (j0 + j >= ti.nvalid) break;
                const int r = ti.r0 + j0 + j;
                const moe_dispatch_meta m = P.meta[P.expert_rows[r]];
                const long long tj = ((long long)m.src_rank * P.lb + m.batch_slot) * P.k + m.route_slot;
                const float y = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), P.s_row[r]), sd);
                if (chok)
                    reinterpret_cast<__nv_bfloat16*>(P.cbuf + tj * P.crow)[ch] = __float2bfloat16_rn(y);
            }
        }
    }
    return true;
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    float* xch = reinterpret_cast<float*>(smem + NS * STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * STAGE_BYTES + XCH_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    auto full = [&](int s) { return bar(s); };
    auto empty = [&](int s) { return bar(NS + s); };
    auto afull = [&](int a) { return bar(2 * NS + a); };
    auto aempty = [&](int a) { return bar(2 * NS + NA + a); };
    auto accfull = [&](int b) { return bar(2 * NS + 2 * NA + b); };
    auto accempty = [&](int b) { return bar(2 * NS + 2 * NA + 2 + b); };
    const uint32_t done_bar = bar(2 * NS + 2 * NA + 4);
    const uint32_t wg_bar = bar(2 * NS + 2 * NA + 5);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int a = 0; a < NA; ++a) {
            ptx::mbar_init(afull(a), 4);
            ptx::mbar_init(aempty(a), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull(b), 1);
            ptx::mbar_init(accempty(b), 4);
        }
        ptx::mbar_init(done_bar, 1);
        ptx::mbar_init(wg_bar, 4);
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmW);
        ptx::prefetch_tmap(&tmX);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int total_tiles = P.tile_prefix[P.G] * P.mb_count;
    const int KS = P.K / BK;
    const int nchunks = (KS + CK - 1) / CK;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const TileInfo ti = decode(P, tile);
                const int yw0 = ti.set * P.rows_per_set + (EPI == EPI_SWIGLU ? ti.mb * 64 : ti.mb * 128);
                const int yw1 = yw0 + P.box1_off;
                for (int ks = 0; ks < KS; ++ks) {
                    const int s = g % NS;
                    if (!ptx::mbar_wait(empty(s), ((g / NS) & 1) ^ 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = ptx::smem_addr(stages + s * STAGE_BYTES);
                    ptx::mbar_expect_tx(full(s), STAGE_BYTES);
                    ptx::tma_load_2d(st, &tmX, ks * BK, ti.r0, full(s));
                    ptx::tma_load_2d(st + B_BYTES, &tmW, ks * BK, yw0, full(s));
                    ptx::tma_load_2d(st + B_BYTES + 4096, &tmW, ks * BK, yw1, full(s));
                    ++g;
                }
            }
            if (!ok) {  // let the loads already issued land before leaving
                for (uint32_t j = (g > NS ? g - NS : 0); j < g; ++j)
                    mbar_wait_quiet(full(j % NS), (j / NS) & 1, DRAIN_NS);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t g = 0, q = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const TileInfo ti = decode(P, tile);
                const uint32_t idesc = ptx::idesc_f16_f32(128, ti.nmma);
                for (int ks = 0; ks < KS; ++ks) {
                    const bool first = (ks % CK) == 0;
                    const bool last = (ks % CK) == CK - 1 || ks == KS - 1;
                    const uint32_t b = q & 1;
                    if (first) {
                        if (!ptx::mbar_wait(accempty(b), ((q >> 1) & 1) ^ 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                    }
                    const int s = g % NS, a = g % NA;
                    if (!ptx::mbar_wait(full(s), (g / NS) & 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT) ||
                        !ptx::mbar_wait(afull(a), (g / NA) & 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t bbase = ptx::smem_addr(stages + s * STAGE_BYTES);
                    const uint32_t d = tmem + TM_ACC + b * 128;
                    const uint32_t abase = tmem + TM_A + a * 32;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx::mma_f16_ts(d, abase + kk * 8, ptx::sdesc_k_sw128(bbase + kk * 32), idesc,
                                        (first && kk == 0) ? 0u : 1u);
                    ptx::tc_commit(empty(s));
                    ptx::tc_commit(aempty(a));
                    if (last) {
                        ptx::tc_commit(accfull(b));
                        ++q;
                    }
                    ++g;
                }
            }
            // every MMA issued above must be complete before TMEM is freed
            ptx::tc_commit(done_bar);
            mbar_wait_quiet(done_bar, 0, WAIT_NS);
        }
    } else {
        // ------------------------- converter / chunk drain / epilogue
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        uint32_t g = 0, q = 0;
        bool ok = true;
        WgBarrier wg{wg_bar, 0};
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
            const TileInfo ti = decode(P, tile);
            const int nsl = (ti.nmma + 31) / 32;

            auto drain = [&](int c, bool final_chunk) -> bool {
                const uint32_t b = q & 1;
                if (!warp_wait(accfull(b), (q >> 1) & 1, P.err)) return false;
                ptx::tc_fence_after();
                const uint32_t accb = tmem + lane_base + TM_ACC + b * 128;
                const uint32_t sumb = tmem + lane_base + TM_SUM;
                for (int sl = 0; sl < nsl; ++sl) {
                    uint32_t v[32], sv[32];
                    ptx::tmem_ld32(accb + sl * 32, v);
                    if (c > 0) ptx::tmem_ld32(sumb + sl * 32, sv);
                    ptx::tmem_wait_ld();
                    int iv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        iv[j] = __float2int_rn(__uint_as_float(v[j])) + (c > 0 ? static_cast<int>(sv[j]) : 0);
                    if (!final_chunk) {
                        uint32_t w[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) w[j] = static_cast<uint32_t>(iv[j]);
                        ptx::tmem_st32(sumb + sl * 32, w);
                    } else if (!epilogue_slice<EPI>(P, ti, row, sl * 32, iv, xch, wg, lane)) {
                        return false;
                    }
                }
                if (!final_chunk) ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(accempty(b));
                ++q;
                return true;
            };

            int next_drain = 0;
            for (int ks = 0; ks < KS; ++ks) {
                const int s = g % NS, a = g % NA;
                if (!warp_wait(full(s), (g / NS) & 1, P.err) ||
                    !warp_wait(aempty(a), ((g / NA) & 1) ^ 1, P.err)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // this thread's weight row: 64 int8 in 64-byte swizzled rows
                const uint8_t* arow = stages + s * STAGE_BYTES + B_BYTES + (row >> 6) * 4096 + (row & 63) * 64;
                const int sw = (row >> 1) & 3;
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(arow + ((c ^ sw) << 4));
                    s8x4_to_f16x4(w.x, v[8 * c + 0], v[8 * c + 1]);
                    s8x4_to_f16x4(w.y, v[8 * c + 2], v[8 * c + 3]);
                    s8x4_to_f16x4(w.z, v[8 * c + 4], v[8 * c + 5]);
                    s8x4_to_f16x4(w.w, v[8 * c + 6], v[8 * c + 7]);
                }
                ptx::tmem_st32(tmem + lane_base + TM_A + a * 32, v);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(afull(a));
                ++g;
                if (next_drain < nchunks - 1 && ks == (next_drain + 1) * CK + NA - 1) {
                    if (!drain(next_drain, false)) {
                        ok = false;
                        break;
                    }
                    ++next_drain;
                }
            }
            while (ok && next_drain < nchunks) {
                if (!drain(next_drain, next_drain == nchunks - 1)) ok = false;
                ++next_drain;
            }
        }
    }

    // ------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------ helpers
// Gather rows (optionally through row_index) of an int8 matrix and convert
// them to fp16 (exact); optionally copy the dispatch scale of each row.
__global__ void __launch_bounds__(128)
assemble_kernel(int K, const int32_t* __restrict__ row_index, const int8_t* __restrict__ A,
                long long lda, const moe_dispatch_meta* __restrict__ meta, __half* __restrict__ out,
                float* __restrict__ s_row) {
    const int r = blockIdx.x;
    const long long g = row_index ? row_index[r] : r;
    const uint4* src = reinterpret_cast<const uint4*>(A + g * lda);
    uint4* dst = reinterpret_cast<uint4*>(out + (long long)r * K);
    for (int c = threadIdx.x; c < K / 16; c += blockDim.x) {
        const uint4 w = __ldg(src + c);
        uint4 o0, o1;
        s8x4_to_f16x4(w.x, o0.x, o0.y);
        s8x4_to_f16x4(w.y, o0.z, o0.w);
        s8x4_to_f16x4(w.z, o1.x, o1.y);
        s8x4_to_f16x4(w.w, o1.z, o1.w);
        dst[2 * c] = o0;
        dst[2 * c + 1] = o1;
    }
    if (meta && threadIdx.x == 0) s_row[r] = meta[g].scale;
}

// Token-wise requantisation of the SwiGLU output h (absmax already reduced
// into rowmax): hq as exact fp16 integers, s_h per row.
__global__ void __launch_bounds__(256)
requant_kernel(int I, const float* __restrict__ h, const unsigned* __restrict__ rowmax,
               __half* __restrict__ hq, float* __restrict__ sh) {
    const int r = blockIdx.x;
    const float s = row_scale(__uint_as_float(rowmax[r]));
    const float4* src = reinterpret_cast<const float4*>(h + (long long)r * I);
    uint2* dst = reinterpret_cast<uint2*>(hq + (long long)r * I);
    for (int c = threadIdx.x; c < I / 4; c += blockDim.x) {
        const float4 v = src[c];
        int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
        if (s != 0.f) {
            q0 = quant1(v.x, s); q1 = quant1(v.y, s); q2 = quant1(v.z, s); q3 = quant1(v.w, s);
        }
        __half2 a = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
        __half2 b = __halves2half2(__int2half_rn(q2), __int2half_rn(q3));
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&a);
        o.y = *reinterpret_cast<uint32_t*>(&b);
        dst[c] = o;
    }
    if (threadIdx.x == 0) sh[r] = s;
}

// INT8 return message: token-wise codes of y into the combine row (t, j).
__global__ void __launch_bounds__(256)
retquant_kernel(int H, int k, int lb, long long crow, const float* __restrict__ y,
                const unsigned* __restrict__ rowmax, const int32_t* __restrict__ expert_rows,
                const moe_dispatch_meta* __restrict__ meta, unsigned char* __restrict__ cbuf,
                float* __restrict__ cscale) {
    const int r = blockIdx.x;
    const moe_dispatch_meta m = meta[expert_rows[r]];
    const long long tj = ((long long)m.src_rank * lb + m.batch_slot) * k + m.route_slot;
    const float s = row_scale(__uint_as_float(rowmax[r]));
    const float4* src = reinterpret_cast<const float4*>(y + (long long)r * H);
    uint32_t* dst = reinterpret_cast<uint32_t*>(cbuf + tj * crow);
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
        const float4 v = src[c];
        uint32_t w = 0;
        if (s != 0.f) {
            w = (uint32_t)(quant1(v.x, s) & 0xff) | ((uint32_t)(quant1(v.y, s) & 0xff) << 8) |
                ((uint32_t)(quant1(v.z, s) & 0xff) << 16) | ((uint32_t)(quant1(v.w, s) & 0xff) << 24);
        }
        dst[c] = w;
    }
    if (threadIdx.x == 0) cscale[tj] = s;
}

// ---------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
              uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * (uint64_t)esize};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

template <int EPI>
cudaError_t launch_gemm(const Params& P, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    gemm_tc_kernel<EPI><<<sm_count(), THREADS, SMEM_BYTES, st>>>(w, x, P);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace tc

// Exact grouped int8 GEMM with int32 output on the tensor-core path.
// Workspace: [status 256 B][tile prefix][fp16 copy of the A rows].
cudaError_t launch_grouped_gemm_tc(int n_groups, const int32_t* offsets, long long max_rows,
                                   const int32_t* row_index, const int8_t* A, long long lda,
                                   const int8_t* B, int N, int K, int32_t* C, void* ws,
                                   cudaStream_t st) {
    using namespace tc;
    char* w = static_cast<char*>(ws);
    int* err = reinterpret_cast<int*>(w);
    int32_t* tp = reinterpret_cast<int32_t*>(w + 256);
    __half* a16 = reinterpret_cast<__half*>(w + 256 + align_up(4LL * (n_groups + 1), 256));
    cudaError_t e = cudaMemsetAsync(err, 0, 256, st);
    if (e != cudaSuccess) return e;
    count_launches(1);
    if ((e = launch_tile_prefix(n_groups, BN, offsets, tp, st)) != cudaSuccess) return e;
    assemble_kernel<<<(unsigned)max_rows, 128, 0, st>>>(K, row_index, A, lda, nullptr, a16, nullptr);
    count_launches(1);
    CUtensorMap mw, mx;
    if (!make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, (uint64_t)n_groups * N, 64, 64,
                  CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a16, K, (uint64_t)max_rows, 64, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    Params P = {};
    P.G = n_groups; P.offsets = offsets; P.tile_prefix = tp; P.g2s = nullptr;
    P.K = K; P.rows_per_set = N; P.nout = N; P.mb_count = (N + 127) / 128; P.box1_off = 64;
    P.c_i32 = C; P.err = err;
    return launch_gemm<EPI_I32>(P, mw, mx, st);
}

bool ffn_tc_eligible(const Dims& d) { return d.H % 64 == 0 && d.I % 64 == 0; }

cudaError_t launch_ffn_tc(const Dims& d, const void* dbuf, long long meta_off,
                          const int32_t* expert_offsets, const int32_t* expert_rows,
                          const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                          const WsLayout& wl, cudaStream_t st) {
    using namespace tc;
    const long long M = (long long)d.T * d.k;
    const moe_dispatch_meta* meta =
        reinterpret_cast<const moe_dispatch_meta*>(static_cast<const char*>(dbuf) + meta_off);
    int* err = ws_ptr<int>(ws, 0);
    int32_t* tp = ws_ptr<int32_t>(ws, wl.tiles);
    unsigned* hmax = ws_ptr<unsigned>(ws, wl.rowmax);
    unsigned* ymax = hmax + M;
    float* s_row = ws_ptr<float>(ws, wl.s_row);
    float* sh = ws_ptr<float>(ws, wl.sh);
    __half* a16 = ws_ptr<__half>(ws, wl.a16);
    float* hbuf = ws_ptr<float>(ws, wl.hbuf);
    __half* hq16 = ws_ptr<__half>(ws, wl.hq16);
    float* ybuf = ws_ptr<float>(ws, wl.ybuf);
    unsigned char* cb = static_cast<unsigned char*>(cbuf);
    const int int8_ret = d.cfmt == MOE_MSG_INT8;
    const int E_w = w.n_sets;
    cudaError_t e;

    if ((e = cudaMemsetAsync(err, 0, 256, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(hmax, 0, sizeof(unsigned) * 2 * M, st)) != cudaSuccess) return e;
    count_launches(2);
    if ((e = launch_tile_prefix(d.E_phys, BN, expert_offsets, tp, st)) != cudaSuccess) return e;
    assemble_kernel<<<(unsigned)M, 128, 0, st>>>(d.H, expert_rows, static_cast<const int8_t*>(dbuf),
                                                 d.drow, meta, a16, s_row);
    count_launches(1);

    CUtensorMap mwgu, mx1, mwd, mx2;
    if (!make_map(&mwgu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.w_gate_up, d.H, (uint64_t)E_w * 2 * d.I,
                  64, 64, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mx1, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a16, d.H, (uint64_t)M, 64, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mwd, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w.w_down, d.I, (uint64_t)E_w * d.H, 64, 64,
                  CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mx2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hq16, d.I, (uint64_t)M, 64, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    Params P1 = {};
    P1.G = d.E_phys; P1.offsets = expert_offsets; P1.tile_prefix = tp; P1.g2s = w.phys_to_weight;
    P1.K = d.H; P1.rows_per_set = 2 * d.I; P1.nout = d.I; P1.mb_count = d.I / 64; P1.box1_off = d.I;
    P1.s_row = s_row; P1.s_ch = w.s_gate_up; P1.out_f32 = hbuf; P1.rowmax = hmax; P1.err = err;
    if ((e = launch_gemm<EPI_SWIGLU>(P1, mwgu, mx1, st)) != cudaSuccess) return e;

    requant_kernel<<<(unsigned)M, 256, 0, st>>>(d.I, hbuf, hmax, hq16, sh);
    count_launches(1);

    Params P2 = {};
    P2.G = d.E_phys; P2.offsets = expert_offsets; P2.tile_prefix = tp; P2.g2s = w.phys_to_weight;
    P2.K = d.I; P2.rows_per_set = d.H; P2.nout = d.H; P2.mb_count = (d.H + 127) / 128; P2.box1_off = 64;
    P2.s_row = sh; P2.s_ch = w.s_down; P2.err = err;
    if (int8_ret) {
        P2.out_f32 = ybuf; P2.rowmax = ymax;
        if ((e = launch_gemm<EPI_DOWN_F32>(P2, mwd, mx2, st)) != cudaSuccess) return e;
        retquant_kernel<<<(unsigned)M, 256, 0, st>>>(d.H, d.k, d.lb, d.crow, ybuf, ymax, expert_rows,
                                                     meta, cb, reinterpret_cast<float*>(cb + scale_off));
        count_launches(1);
    } else {
        P2.expert_rows = expert_rows; P2.meta = meta; P2.cbuf = cb; P2.crow = d.crow; P2.k = d.k; P2.lb = d.lb;
        if ((e = launch_gemm<EPI_DOWN_BF16>(P2, mwd, mx2, st)) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace moe
