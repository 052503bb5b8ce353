// ffn.cu -- grouped W8A8 SwiGLU expert FFN.
//
// "xDeepServe on CloudMatrix384", section "DeepSeek INT8 量化": P085 (token-wise
// activation scales, channel-wise weight scales, y_ij ~ s_i s^w_j
// sum_k q(x_ik) q(w_jk) on the INT8 matmul unit), P088 (up_proj and gate_proj
// fused into one kernel), P089 (expert inputs and outputs are INT8 in
// communication).  "CloudMatrix384 LLM Serving", section "EP320：token 去找专家"
// (assemble_expert_inputs / run_local_experts / remote_write_combine by
// (source_rank, batch_slot, route_slot)).
//
// Steps (one stream):
//   tiles      per-expert M-tile prefix sums (one block)
//   gemm       C[r][n] = sum_k A[row(r)][k] * B[set(p)][n][k]   exact int32
//              (gate/up: A = dispatch codes gathered by expert_rows, N = 2I)
//   swiglu     g, u -> h = SiLU(g) u -> token-wise INT8 requantisation
//   gemm       down projection, A = requantised rows, N = H
//   ret        y = (acc * s_h) * sd -> return message into the combine
//              buffer at (t, j) (INT8 codes + scale, or bf16)
#include <cuda_bf16.h>

#include "device_math.cuh"
#include "internal.cuh"

namespace moe {
namespace {

// --------------------------------------------------------- tile prefix
// tile_prefix[g] = sum_{g' < g} ceil(M_g' / BM), g = 0..G (one block); BM is
// a multiple of 16.  With a non-null `table`, entry tile_prefix[g] + j
// describes token tile j of group g: (weight set, first row, rows, g).
// The offsets and weight sets are caller data.  Unless offsets[0] = 0, the
// offsets never decrease, offsets[G] <= max_rows and every weight set lies in
// [0, n_sets), the kernel posts MOE_ERR_INDEX and describes no tile at all,
// so no GEMM that reads this prefix addresses memory outside its buffers.
// Groups with 1..skip_rows rows get no tile; with a non-null `narrow`, their
// ids are listed in ascending order in narrow[1..] and their number in
// narrow[0] (for the kernels that take them).
__global__ void __launch_bounds__(1024)
tile_prefix_kernel(int G, int BM, const int32_t* __restrict__ offsets, long long max_rows,
                   int n_sets, int32_t* __restrict__ tile_prefix, int4* __restrict__ table,
                   const int32_t* __restrict__ g2s, int* __restrict__ err, int skip_rows,
                   int32_t* __restrict__ narrow) {
    __shared__ int s_warp[32], s_nwarp[32];
    __shared__ int s_carry, s_ncarry;
    int bad = 0;
    for (int g = threadIdx.x; g < G; g += 1024) {
        if (offsets[g + 1] < offsets[g]) bad = 1;
        const int set = g2s ? g2s[g] : g;
        if (set < 0 || set >= n_sets) bad = 1;
    }
    if (threadIdx.x == 0 && (offsets[0] != 0 || (long long)offsets[G] > max_rows)) bad = 1;
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0 && err) post_status(err, MOE_ERR_INDEX);
        for (int g = threadIdx.x; g <= G; g += 1024) tile_prefix[g] = 0;
        if (threadIdx.x == 0 && narrow) narrow[0] = 0;
        return;
    }
    if (threadIdx.x == 0) {
        s_carry = 0;
        s_ncarry = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int b0 = 0; b0 < G; b0 += 1024) {
        int g = b0 + threadIdx.x;
        int n = 0, nf = 0;
        if (g < G) {
            int m = offsets[g + 1] - offsets[g];
            n = m > skip_rows ? (m + BM - 1) / BM : 0;  // narrow groups: no tile here
            nf = m >= 1 && m <= skip_rows;
        }
        int v = n, vn = nf;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, v, off);
            int on = __shfl_up_sync(0xffffffffu, vn, off);
            if (lane >= off) {
                v += o;
                vn += on;
            }
        }
        if (lane == 31) {
            s_warp[w] = v;
            s_nwarp[w] = vn;
        }
        __syncthreads();
        if (w == 0) {
            int x = s_warp[lane], xn = s_nwarp[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int o = __shfl_up_sync(0xffffffffu, x, off);
                int on = __shfl_up_sync(0xffffffffu, xn, off);
                if (lane >= off) {
                    x += o;
                    xn += on;
                }
            }
            s_warp[lane] = x;
            s_nwarp[lane] = xn;
        }
        __syncthreads();
        int incl = v + (w > 0 ? s_warp[w - 1] : 0) + s_carry;
        const int nincl = vn + (w > 0 ? s_nwarp[w - 1] : 0) + s_ncarry;
        if (narrow && nf) narrow[1 + nincl - 1] = g;
        if (g < G) {
            tile_prefix[g] = incl - n;
            if (table) {
                // the group's rows split evenly over its n tiles in units of
                // 16 rows (the MMA's N step): u or u + 1 units a tile, at
                // most BM rows, the last tile holding the remainder, so only
                // it rounds its rows up, not n - 1 full tiles and a ragged one
                const int r0 = offsets[g], m = offsets[g + 1] - r0;
                const int set = g2s ? g2s[g] : g;
                const int units = (m + 15) / 16;
                const int u = n > 0 ? units / n : 0, extra = units - u * n;
                for (int j = 0; j < n; ++j) {
                    const int start = 16 * (j * u + min(j, extra));
                    const int rows = min(16 * (u + (j < extra ? 1 : 0)), m - start);
                    table[incl - n + j] = make_int4(set, r0 + start, rows, g);
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 1023) {
            s_carry = incl;
            s_ncarry = nincl;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        tile_prefix[G] = s_carry;
        if (narrow) narrow[0] = s_ncarry;
    }
}

// ------------------------------------------------------- SIMT int8 GEMM
// 64x64 output tile per 256-thread block, K in 64-byte steps, dp4a
// (4 int8 products summed into int32, exact).
constexpr int kBM = 64, kBN = 64, kBKW = 16;  // BK = 64 bytes = 16 words

__global__ void __launch_bounds__(256)
gemm_s8_simt_kernel(int G, const int32_t* __restrict__ offsets,
                    const int32_t* __restrict__ tile_prefix, const int32_t* __restrict__ row_index,
                    long long a_rows, const int8_t* __restrict__ A, long long lda,
                    const int8_t* __restrict__ B, long long bstride, const int32_t* __restrict__ g2s,
                    int N, int K, int32_t* __restrict__ C, int* __restrict__ err) {
    __shared__ int As[kBM][kBKW + 1];
    __shared__ int Bs[kBN][kBKW + 1];
    const int tile = blockIdx.x;
    if (tile >= tile_prefix[G]) return;
    const int g = find_group(tile_prefix, G, tile);
    const int m0 = offsets[g] + (tile - tile_prefix[g]) * kBM;
    const int mend = offsets[g + 1];
    const int n0 = blockIdx.y * kBN;
    const int set = g2s ? g2s[g] : g;
    const int8_t* Bg = B + (long long)set * bstride;

    const int tid = threadIdx.x;
    const int lr = tid >> 2, lq = tid & 3;  // load row, 16-byte quarter
    bool a_ok = m0 + lr < mend;
    long long arow = 0;
    if (a_ok) arow = row_index ? row_index[m0 + lr] : (m0 + lr);
    if (a_ok && (arow < 0 || arow >= a_rows)) {  // row list entry outside A: read zeros
        post_status(err, MOE_ERR_INDEX);
        a_ok = false;
        arow = 0;
    }
    const int8_t* ap = A + arow * lda + lq * 16;
    const bool b_ok = n0 + lr < N;
    const int8_t* bp = Bg + (long long)(n0 + lr) * K + lq * 16;

    const int ty = tid >> 4, tx = tid & 15;
    int acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0;

    for (int k0 = 0; k0 < K; k0 += 64) {
        const bool kin = k0 + lq * 16 < K;
        int4 va = make_int4(0, 0, 0, 0), vb = make_int4(0, 0, 0, 0);
        if (a_ok && kin) va = __ldg(reinterpret_cast<const int4*>(ap + k0));
        if (b_ok && kin) vb = __ldg(reinterpret_cast<const int4*>(bp + k0));
        As[lr][lq * 4 + 0] = va.x; As[lr][lq * 4 + 1] = va.y;
        As[lr][lq * 4 + 2] = va.z; As[lr][lq * 4 + 3] = va.w;
        Bs[lr][lq * 4 + 0] = vb.x; Bs[lr][lq * 4 + 1] = vb.y;
        Bs[lr][lq * 4 + 2] = vb.z; Bs[lr][lq * 4 + 3] = vb.w;
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBKW; ++kk) {
            int a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[ty * 4 + i][kk];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[tx * 4 + j][kk];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __dp4a(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int m = m0 + ty * 4 + i;
        if (m >= mend) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int n = n0 + tx * 4 + j;
            if (n < N) C[(long long)m * N + n] = acc[i][j];
        }
    }
}

// ----------------------------------------------------- block reductions
template <int NT>
__device__ __forceinline__ float block_max(float v, float* s_red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = s_red[0];
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) r = fmaxf(r, s_red[i]);
    __syncthreads();
    return r;
}

constexpr int kRowThreads = 256;

// SwiGLU + token-wise requantisation of one routed row.
__global__ void __launch_bounds__(kRowThreads)
swiglu_requant_kernel(int I, int E_phys, int n_sets, long long nslots,
                      const int32_t* __restrict__ expert_offsets,
                      const int32_t* __restrict__ expert_rows,
                      const moe_dispatch_meta* __restrict__ meta,
                      const int32_t* __restrict__ p2w, const float* __restrict__ s_gu,
                      const int32_t* __restrict__ acc_gu, int8_t* __restrict__ hq,
                      float* __restrict__ sh, int* __restrict__ err) {
    extern __shared__ float s_h[];
    __shared__ float s_red[kRowThreads / 32];
    const int r = blockIdx.x;
    const int p = find_group(expert_offsets, E_phys, r);
    const int set = p2w ? p2w[p] : p;
    const long long g = expert_rows[r];
    if (set < 0 || set >= n_sets || g < 0 || g >= nslots) {  // caller data out of range
        if (threadIdx.x == 0) post_status(err, MOE_ERR_INDEX);
        return;
    }
    const float s = meta[g].scale;
    const int32_t* acc = acc_gu + (long long)r * 2 * I;
    const float* sg = s_gu + (long long)set * 2 * I;
    float amax = 0.f;
    for (int i = threadIdx.x; i < I; i += kRowThreads) {
        float gv = __fmul_rn(__fmul_rn(__int2float_rn(acc[i]), s), sg[i]);
        float uv = __fmul_rn(__fmul_rn(__int2float_rn(acc[I + i]), s), sg[I + i]);
        float h = __fmul_rn(silu_spec(gv), uv);
        s_h[i] = h;
        amax = fmaxf(amax, fabsf(h));
    }
    amax = block_max<kRowThreads>(amax, s_red);
    const float sc = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.0f);
    int8_t* out = hq + (long long)r * I;
    for (int i = threadIdx.x; i < I; i += kRowThreads)
        out[i] = (int8_t)(sc == 0.f ? 0 : quant1(s_h[i], sc));
    if (threadIdx.x == 0) sh[r] = sc;
}

// Down-projection epilogue: y, then the return message into the combine row.
__global__ void __launch_bounds__(kRowThreads)
return_kernel(int H, int k, int lb, int S, int E_phys, int n_sets, long long nslots, int int8_msgs,
              long long crow, const int32_t* __restrict__ expert_offsets,
              const int32_t* __restrict__ expert_rows,
              const moe_dispatch_meta* __restrict__ meta, const int32_t* __restrict__ p2w,
              const float* __restrict__ s_d, const int32_t* __restrict__ acc_d,
              const float* __restrict__ sh, unsigned char* __restrict__ cbuf,
              float* __restrict__ cscale, int* __restrict__ err) {
    extern __shared__ float s_y[];
    __shared__ float s_red[kRowThreads / 32];
    const int r = blockIdx.x;
    const int p = find_group(expert_offsets, E_phys, r);
    const int set = p2w ? p2w[p] : p;
    const long long g = expert_rows[r];
    if (set < 0 || set >= n_sets || g < 0 || g >= nslots) {
        if (threadIdx.x == 0) post_status(err, MOE_ERR_INDEX);
        return;
    }
    const moe_dispatch_meta m = meta[g];
    if (!meta_in_range(m, S, lb, k)) {  // the slot holds no message of this shape
        if (threadIdx.x == 0) post_status(err, MOE_ERR_INDEX);
        return;
    }
    const long long tj = ((long long)m.src_rank * lb + m.batch_slot) * k + m.route_slot;
    const int32_t* acc = acc_d + (long long)r * H;
    const float* sd = s_d + (long long)set * H;
    const float shr = sh[r];
    unsigned char* row = cbuf + tj * crow;
    float amax = 0.f;
    for (int c = threadIdx.x; c < H; c += kRowThreads) {
        float y = __fmul_rn(__fmul_rn(__int2float_rn(acc[c]), shr), sd[c]);
        if (int8_msgs) {
            s_y[c] = y;
            amax = fmaxf(amax, fabsf(y));
        } else {
            reinterpret_cast<__nv_bfloat16*>(row)[c] = __float2bfloat16_rn(y);
        }
    }
    if (!int8_msgs) return;
    amax = block_max<kRowThreads>(amax, s_red);
    const float sc = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.0f);
    for (int c = threadIdx.x; c < H; c += kRowThreads)
        reinterpret_cast<int8_t*>(row)[c] = (int8_t)(sc == 0.f ? 0 : quant1(s_y[c], sc));
    if (threadIdx.x == 0) cscale[tj] = sc;
}

cudaError_t set_smem(const void* fn, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_tile_prefix(int G, int BM, const int32_t* offsets, long long max_rows, int n_sets,
                               int32_t* tile_prefix, int* err, cudaStream_t st, int4* table,
                               const int32_t* g2s, int skip_rows, int32_t* narrow) {
    tile_prefix_kernel<<<1, 1024, 0, st>>>(G, BM, offsets, max_rows, n_sets, tile_prefix, table, g2s,
                                           err, skip_rows, narrow);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_s8(int n_groups, const int32_t* offsets, long long max_rows,
                                   const int32_t* row_index, long long a_rows, const int8_t* A,
                                   long long lda, const int8_t* B, long long b_group_stride,
                                   const int32_t* group_to_set, int n_sets, int N, int K, int32_t* C,
                                   int32_t* tile_prefix, int* err, cudaStream_t st) {
    cudaError_t e0 = launch_tile_prefix(n_groups, kBM, offsets, max_rows, n_sets, tile_prefix, err, st,
                                        nullptr, group_to_set);
    if (e0 != cudaSuccess) return e0;
    long long max_tiles = (max_rows + kBM - 1) / kBM + n_groups;
    if (max_tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid((unsigned)max_tiles, (unsigned)((N + kBN - 1) / kBN));
    gemm_s8_simt_kernel<<<grid, 256, 0, st>>>(n_groups, offsets, tile_prefix, row_index, a_rows, A,
                                              lda, B, b_group_stride, group_to_set, N, K, C, err);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_ffn_simt(const Dims& d, const void* dbuf, long long meta_off,
                            const int32_t* expert_offsets, const int32_t* expert_rows,
                            const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear) {
    const long long M = (long long)d.T * d.k;
    const moe_dispatch_meta* meta =
        reinterpret_cast<const moe_dispatch_meta*>(static_cast<const char*>(dbuf) + meta_off);
    int32_t* tiles = ws_ptr<int32_t>(ws, wl.tiles);
    int32_t* acc_gu = ws_ptr<int32_t>(ws, wl.acc_gu);
    int8_t* hq = ws_ptr<int8_t>(ws, wl.hq);
    float* sh = ws_ptr<float>(ws, wl.sh);
    int32_t* acc_d = ws_ptr<int32_t>(ws, wl.acc_d);
    unsigned char* cb = static_cast<unsigned char*>(cbuf);
    cudaError_t e;

    int* err = ws_ptr<int>(ws, 0);
    if (clear && (e = clear_status(ws, st)) != cudaSuccess) return e;
    e = launch_grouped_gemm_s8(d.E_phys, expert_offsets, M, expert_rows, d.nslots,
                               static_cast<const int8_t*>(dbuf), d.drow, w.w_gate_up,
                               2LL * d.I * d.H, w.phys_to_weight, w.n_sets, 2 * d.I, d.H, acc_gu,
                               tiles, err, st);
    if (e != cudaSuccess) return e;
    size_t sm1 = sizeof(float) * (size_t)d.I;
    if ((e = set_smem((const void*)swiglu_requant_kernel, sm1)) != cudaSuccess) return e;
    swiglu_requant_kernel<<<(unsigned)M, kRowThreads, sm1, st>>>(
        d.I, d.E_phys, w.n_sets, d.nslots, expert_offsets, expert_rows, meta, w.phys_to_weight,
        w.s_gate_up, acc_gu, hq, sh, err);
    e = launch_grouped_gemm_s8(d.E_phys, expert_offsets, M, nullptr, M, hq, d.I, w.w_down,
                               (long long)d.H * d.I, w.phys_to_weight, w.n_sets, d.H, d.I, acc_d,
                               tiles, err, st);
    if (e != cudaSuccess) return e;
    const int int8_msgs = d.cfmt == MOE_MSG_INT8 ? 1 : 0;
    size_t sm2 = int8_msgs ? sizeof(float) * (size_t)d.H : 0;
    if ((e = set_smem((const void*)return_kernel, sm2)) != cudaSuccess) return e;
    return_kernel<<<(unsigned)M, kRowThreads, sm2, st>>>(
        d.H, d.k, d.lb, d.S, d.E_phys, w.n_sets, d.nslots, int8_msgs, d.crow, expert_offsets,
        expert_rows, meta, w.phys_to_weight, w.s_down, acc_d, sh, cb,
        reinterpret_cast<float*>(cb + scale_off), err);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace moe
