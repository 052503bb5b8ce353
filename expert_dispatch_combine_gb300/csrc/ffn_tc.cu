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
// kind::f16: every int8 value is exact in fp16, every product (|p| <= 16384)
// is exact in fp32, and the fp32 accumulator is drained to int32 every 1024
// K (1024 * 16384 = 2^24, so every partial sum is an exact integer).  The
// int32 results equal the integer matrix product bit for bit.
//
// GEMM structure (one CTA per SM, persistent over tiles):
//   D^T[channel][token] = W[channel][:] . X[token][:]
//   A operand = weights, 128 channel rows per tile, in one of two forms:
//     int8 (the layer's weights): TMA loads int8 tiles into shared memory; a
//     converter warpgroup turns them into fp16 and stores them in tensor
//     memory (the A-from-TMEM form of tcgen05.mma);
//     fp16 copies (made once by moe_weights_to_f16, twice the bytes): TMA
//     loads them straight into shared memory and the MMA reads both operands
//     from there (the SS form); no conversion on the SM, 256-token tiles, run
//     by CTA pairs (cta_group::2: a cluster of two CTAs computes 256 channels
//     of a tile with M = 256 MMAs issued by the even CTA, each CTA staging its
//     own 128 weight rows and half of the tokens);
//   B operand = activations, up to BN tokens per tile (fp16, K-major, 128B
//     swizzle), TMA-loaded in 32-row boxes so that small experts only load
//     the rows they have; the MMA N is the tile's token count rounded up to 16.
//   TMEM (512 columns): two BN-column fp32 accumulators, so that the drain
//     of one 1024-K chunk overlaps the MMAs of the next, and (int8 form) the
//     rest in pairs of 32-column A slots (two pairs at BN = 192, six at the
//     64-token decode tiles).  The int32 running sums live in registers of
//     two drain warpgroups (BN / 2 token columns each).
//   Issue: int8 form, the single MMA thread waits once per PAIR of 64-K
//     stages (8 MMAs): each wait costs the issuing thread a few hundred
//     cycles, which 4 MMAs of N <= 224 do not cover but 8 do, and the
//     converter fills the A slots of one pair while the MMAs of the others
//     run; fp16 form on CTA pairs, one wait per pair of 32 KB stages (8 M =
//     256 MMAs, three ring slots).  The MMA thread's per-wait cost bounds the
//     pipeline (one 64-K stage took about 340 ns whatever the tile on a single
//     CTA, one wait per 48 KB stage); the pair does twice the tensor work per
//     wait and stage.
//   Epilogue: each 16-token group is scaled, staged in shared memory and
//     written with one TMA tensor store (partial groups use plain stores).
// The gate/up GEMM computes the gate and up projections g, u of all 2I
// channels in one launch (P088) and writes them as f32; SwiGLU h = SiLU(g) u,
// its row maximum and the token-wise requantisation run in one row kernel
// (requant_kernel), so the SiLU's instructions stay off the GEMM's critical
// path.  The down GEMM's epilogue writes y and reduces its row maximum.
// Warp roles (16 warps): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 4-7 converter (idle with fp16 weights), warps 8-15 two drain/epilogue
// warpgroups.  Tiles run in raster bands (tile_entry) so that the CTAs that
// share a weight block start together.  Register
// budgets are moved between warpgroups with setmaxnreg (the totals stay
// within the launch allocation).  Each warpgroup covers the four TMEM lane
// quarters.
// Every mbarrier wait is bounded (2 s): on a timeout the kernel records
// MOE_ERR_TIMEOUT in the workspace status word, waits briefly for its own
// copies in flight, frees TMEM and returns.
#include <algorithm>
#include <climits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "combine_math.cuh"
#include "device_math.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BK = 64;                           // K per stage
constexpr int CK = 16;                           // stages per exact chunk (1024 K)
constexpr int BOX_ROWS = 32;                     // token rows per activation TMA box
constexpr int BOX_BYTES = BOX_ROWS * BK * 2;     // 4 KB
constexpr int GT = 16;                           // tokens per epilogue group
constexpr int STG_BYTES = GT * 128 * 4;          // 8 KB staging buffer; two per drain warpgroup
constexpr uint32_t TM_ACC = 0, TM_COLS = 512;
constexpr int THREADS = 512;

// Shapes that depend on the tile's token count BN and on the weight operand.
// int8 weights (AF16 false), converted on the SM: BN 192 for batches with
// many rows per expert, 64 for decode-sized batches, where the smaller
// activation region buys twice the stages (weight bytes in flight).  The
// TMEM columns after the two accumulators hold NAP pairs of A slots (64
// columns per stage pair): the converter can fill pair p while the MMAs of
// pairs p - NAP + 1 .. p - 1 run.  More A pairs than shared-memory pairs
// would never be used.
// fp16 copies of the int8 weights (AF16 true): both operands are read from
// shared memory by the MMA, no A slots.  The stage ring is latency-bound
// (about 192 KB in flight per SM against L2/DRAM latency), so the widest tile
// wins: BN 256 with four 48 KB stages (measured 0.84 of the bf16 peak on 1024
// rows per expert, against 0.76 / 0.67 / 0.58 / 0.49 at BN 224 / 192 / 160 /
// 128).
// CTA pairs (PAIR, fp16 weights, 256-token tiles): the two CTAs of a cluster
// run a tile of 256 channels with one M = 256 MMA per K step; each stages its
// own 128 weight rows and half of the tile's tokens, 32 KB a stage, six
// stages in pairs (one wait for 8 MMAs, three ring slots).  The per-stage
// control cost (the MMA thread's wait, issue and commit) bounds the
// single-CTA form; the pair form does twice the tensor work per wait.
template <int BNV, bool AF16 = false, bool PAIR = false>
struct Tile {
    static constexpr int BN = BNV;                            // tokens per tile
    static constexpr int A_BYTES = AF16 ? 128 * BK * 2 : 128 * BK;  // weights per stage (16 / 8 KB)
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;  // this CTA's fp16 activations per stage
    static constexpr int STAGE_BYTES = B_BYTES + A_BYTES;
    // shared-memory stages: for fp16 weights as many as fit beside the
    // epilogue staging buffers and the barriers
    static constexpr int NS_F16 = (227 * 1024 - 4 * STG_BYTES - 2048) / STAGE_BYTES;
    static constexpr int NS = AF16 ? NS_F16 : (BN == 64 ? 12 : 6);
    // stages per pipeline step (one full/empty barrier pair and one wait of
    // the MMA thread per step): pairs for int8 weights and for CTA pairs,
    // single stages for fp16 weights on one CTA, whose 48 KB stages would
    // leave only two pair slots
    static constexpr int SPS = (AF16 && !PAIR) ? 1 : 2;
    static constexpr int NP = NS / SPS;                       // step slots
    static constexpr uint32_t TM_A = 2 * BN;                  // after the two accumulators
    static constexpr int NAP_FIT = (TM_COLS - TM_A) / 64;     // A-slot pairs that fit in TMEM
    static constexpr int NAP = AF16 ? 0 : (NAP_FIT < NP ? NAP_FIT : NP);  // A-slot pairs used
    static constexpr int HALF = BN / 2;                       // token columns per drain warpgroup
    static constexpr int NGRP = HALF / GT;                    // epilogue groups per drain warpgroup
    static constexpr int NAB = NAP > 0 ? NAP : 1;             // A-slot barriers (one unused with fp16 weights)
    static constexpr int NBARS = 2 * NP + NAB + 4 + 1 + 2;
    static constexpr int SMEM_BYTES = NS * STAGE_BYTES + 4 * STG_BYTES + NBARS * 8 + 16 + 1024;
    static_assert(BN % 32 == 0 && BN <= 256 && HALF % GT == 0 && NS % SPS == 0 && CK % SPS == 0, "tile shape");
    static_assert(B_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "operands start on 128B-swizzle atoms");
    static_assert(SMEM_BYTES <= 227 * 1024, "dynamic shared memory per CTA");
    static_assert(!PAIR || (AF16 && BN == 256), "CTA pairs take fp16 weights and 256-token tiles");
    static_assert(AF16 ? TM_A <= TM_COLS : (NAP >= 2 && TM_A + NAP * 64 <= TM_COLS),
                  "two accumulators (and, for int8 weights, two or more A-slot pairs) in TMEM");
};
// the fp16-copy GEMMs run as CTA pairs
constexpr bool kPairF16 = true;
// token tiles per raster band (tile order, below)
constexpr int kRasterTokenTiles = 8;
constexpr int BN_LARGE = kTcTileRows, BN_DECODE = kTcMinTileRows, BN_F16 = kTcTileRowsF16;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 20000000ull;
// per-thread register budgets after setmaxnreg: 128 threads each at
// 48 (producer/MMA) + 96 (converter) + 2 x 184 (drains) = 65,536 <= 512 x 128;
// with fp16 weights the converter warpgroup idles at the minimum, 24, and the
// drains (128 token columns each at BN 256) take 216: 64,512
constexpr uint32_t REG_CTRL = 48, REG_CONV = 96, REG_DRAIN = 184;
constexpr uint32_t REG_IDLE = 24, REG_DRAIN_F16 = 216;
static_assert(128 * (REG_CTRL + REG_CONV + 2 * REG_DRAIN) <= THREADS * 128, "register split");
static_assert(128 * (REG_CTRL + REG_IDLE + 2 * REG_DRAIN_F16) <= THREADS * 128, "register split (fp16 weights)");

enum { EPI_I32 = 0, EPI_GU = 1, EPI_F32 = 2, EPI_BF16MSG = 3 };

struct Params {
    int G;
    const int32_t* offsets;      // [G+1] token rows per group
    const int32_t* tile_prefix;  // [G+1] token tiles per group
    const int4* ttab;            // per token tile: (weight set, first row, rows, group)
    const int32_t* g2s;          // nullable: weight set of each group
    int K;                       // reduction length, multiple of 64
    int rows_per_set;            // weight rows per set
    int nout;                    // output channels per set (EPI_GU: 2I, gate then up)
    int mb_count;                // channel blocks per token tile
    int box1_off;                // row offset of the second 64-row weight box
    const float* s_row;          // per token-row scale
    const float* s_ch;           // per-channel weight scales [set][rows_per_set]
    int32_t* c_i32;              // EPI_I32: [M][nout]
    float* out_f32;              // EPI_GU: g and u [M][2I]; EPI_F32: y [M][nout]
    unsigned* rowmax;            // EPI_F32: per-row absmax of y (float bits)
    const int32_t* expert_rows;  // EPI_BF16MSG: row -> dispatch slot
    const moe_dispatch_meta* meta;
    unsigned char* cbuf;
    long long crow;
    int k, lb, S;
    long long nslots;            // EPI_BF16MSG: dispatch slots (range of expert_rows entries)
    int tma_out;                 // epilogue may use tensor stores for full groups
    int* err;
};

struct TileInfo {
    int set, r0, nvalid, nmma, mb;
};

// Tile order: group by group (group g owns tiles [tp[g], tp[g+1]) * mb_count,
// tp the tile prefix); inside a group, its token tiles in bands of up to
// kRasterTokenTiles, and inside a band channel block by channel block with
// the band's token tiles side by side.  CTAs that start together then share
// each weight block (one DRAM read for the band, taken in step), while a
// band's activations stay few enough to live in L2 across its channel
// blocks.  Each role reads the table entry of its next tile when the current
// one starts.  The entry is three dependent reads, and the role waits for the
// first two in line; spreading all three over earlier tiles measured no faster.
struct TileRef {
    int4 e;  // token-tile table entry
    int mb;  // channel block
};
__device__ __forceinline__ TileRef tile_entry(const Params& P, int tile, int total_tiles) {
    if (tile >= total_tiles) return TileRef{make_int4(0, 0, 0, 0), 0};
    // tile / mb_count is a token tile of the same group (not of this tile)
    const int g = __ldg(P.ttab + tile / P.mb_count).w;
    const int t0 = __ldg(P.tile_prefix + g), nt = __ldg(P.tile_prefix + g + 1) - t0;
    const int local = tile - t0 * P.mb_count;  // in [0, nt * mb_count)
    const int band = local / (kRasterTokenTiles * P.mb_count);
    const int r = local - band * kRasterTokenTiles * P.mb_count;
    const int bs = min(kRasterTokenTiles, nt - band * kRasterTokenTiles);  // token tiles in the band
    const int mb = r / bs;
    return TileRef{__ldg(P.ttab + t0 + band * kRasterTokenTiles + (r - mb * bs)), mb};
}
__device__ __forceinline__ TileInfo decode(const Params& P, int tile, const TileRef& r) {
    const int4& e = r.e;
    TileInfo t;
    t.mb = r.mb;
    t.set = e.x;
    t.r0 = e.y;
    t.nvalid = e.z;
    t.nmma = (t.nvalid + 15) & ~15;
    return t;
}

// Warp-uniform bounded wait: every lane waits (each acquires the phase), and
// the warp goes on only if all lanes saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
    const bool ok = ptx::mbar_wait(bar, parity, err, WAIT_NS, MOE_ERR_TIMEOUT);
    return __all_sync(0xffffffffu, ok);
}

// Bounded barrier of the four warps of one warpgroup (an mbarrier with count
// 4 instead of bar.sync, so that a warp that gave up cannot hang the others).
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

template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Epilogue for one 16-token group of a finished tile with plain stores (used
// for partial groups and for bf16 return messages).  `row` is this thread's
// TMEM lane (weight channel within the tile), iv[j] the exact int32 result
// for token j0 + j.  Per-token values are loaded once per lane and broadcast
// with shuffles.
template <int EPI>
__device__ __forceinline__ void epilogue_direct(const Params& P, const TileInfo& ti, int row,
                                                int lane, int j0, const int (&iv)[GT]) {
    const bool lane_ok = lane < GT && j0 + lane < ti.nvalid;
    if constexpr (EPI == EPI_I32) {
        const int ch = ti.mb * 128 + row;
        if (ch < P.nout) {
#pragma unroll
            for (int j = 0; j < GT; ++j)
                if (j0 + j < ti.nvalid) P.c_i32[(long long)(ti.r0 + j0 + j) * P.nout + ch] = iv[j];
        }
    } else if constexpr (EPI == EPI_GU || EPI == EPI_F32) {
        const int col = ti.mb * 128 + row, ld = P.nout;
        const bool chok = col < P.nout;
        const float sc = chok ? P.s_ch[(long long)ti.set * P.rows_per_set + col] : 0.f;
        const float sr_l = lane_ok ? P.s_row[ti.r0 + j0 + lane] : 0.f;
        float* out = P.out_f32 + (long long)ti.r0 * ld + col;
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            const float sr = __shfl_sync(0xffffffffu, sr_l, j);
            const float v = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), sr), sc);
            if (chok && j0 + j < ti.nvalid) out[(long long)(j0 + j) * ld] = v;
        }
    } else {  // EPI_BF16MSG: the return message is bf16(y), written in place
        const int ch = ti.mb * 128 + row;
        const bool chok = ch < P.nout;
        const float sd = chok ? P.s_ch[(long long)ti.set * P.rows_per_set + ch] : 0.f;
        const float sr_l = lane_ok ? P.s_row[ti.r0 + j0 + lane] : 0.f;
        int tj_l = -1;  // -1: no valid message for this token (slot or metadata out of range)
        if (lane_ok) {
            const long long g = P.expert_rows[ti.r0 + j0 + lane];
            bool ok = g >= 0 && g < P.nslots;
            if (ok) {
                const moe_dispatch_meta m = P.meta[g];
                ok = meta_in_range(m, P.S, P.lb, P.k);
                if (ok) tj_l = (m.src_rank * P.lb + m.batch_slot) * P.k + m.route_slot;
            }
            if (!ok) post_status(P.err, MOE_ERR_INDEX);
        }
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            const float sr = __shfl_sync(0xffffffffu, sr_l, j);
            const int tj = __shfl_sync(0xffffffffu, tj_l, j);
            const float y = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), sr), sd);
            if (chok && j0 + j < ti.nvalid && tj >= 0)
                reinterpret_cast<__nv_bfloat16*>(P.cbuf + (long long)tj * P.crow)[ch] =
                    __float2bfloat16_rn(y);
        }
    }
}

// Epilogue for a full 16-token group through shared memory and one TMA
// tensor store (int32 results).  All four warps of the drain warpgroup take
// part; `leader` issues the store.
template <int EPI>
__device__ __forceinline__ bool epilogue_tma(const Params& P, const TileInfo& ti, int row,
                                             int lane, int j0, const int (&iv)[GT], uint8_t* stg,
                                             const CUtensorMap* tmO, WgBarrier& wg, bool leader) {
    int32_t* o = reinterpret_cast<int32_t*>(stg) + row;
#pragma unroll
    for (int j = 0; j < GT; ++j) o[j * 128] = iv[j];
    ptx::fence_proxy_async_smem();
    if (!wg.sync(lane, P.err)) return false;
    if (leader) {
        ptx::tma_store_2d(tmO, ti.mb * 128, ti.r0 + j0, ptx::smem_addr(stg));
        ptx::bulk_commit();
        ptx::bulk_wait_read0();
    }
    return wg.sync(lane, P.err);  // staging buffer free again
}

// Epilogue of the expert FFN for one 16-token group, staged in shared memory:
// v = (acc * s_row) * s_ch for the tile's 128 channels (EPI_GU: the gate and
// up projections g and u, channels of [2I]; EPI_F32: y).  For EPI_F32 the
// per-row absolute maximum of this tile's outputs also goes to `rowmax` with
// an atomic max (the INT8 return message needs the whole row).  The values go
// out with one TMA tensor store for a full group, plain stores for a partial
// one.  All four warps of the drain warpgroup take part.
// Groups alternate between two staging buffers, with one warpgroup barrier
// per group: every thread's reads of a buffer precede its arrival at the next
// group's barrier, and before that barrier the leader waits for the previous
// group's tensor store to have read its buffer, so a buffer is free again
// when the group after next writes it.
// The token scales of the warpgroup's columns and the channel scale come in
// from the tile's start (srv[q]: token tok0 + 32 q + lane, 0 past the tile's
// rows; sd: 0 past the outputs), so that no group waits on a global load;
// tl0 is the group's first column within the warpgroup's half (a constant
// once the group loop is unrolled).
template <int EPI, int NQ>
__device__ __forceinline__ bool epilogue_staged(const Params& P, const TileInfo& ti, int row,
                                                int lane, int j0, int tl0, const int (&iv)[GT],
                                                const float (&srv)[NQ], float sd, float* stg,
                                                const CUtensorMap* tmO, WgBarrier& wg, bool leader) {
    const int nv = min(GT, ti.nvalid - j0);  // valid tokens in this group (>= 1)
    const int col = ti.mb * 128 + row;
    const bool chok = col < P.nout;
#pragma unroll
    for (int j = 0; j < GT; ++j) {
        const float sr = __shfl_sync(0xffffffffu, srv[(tl0 + j) >> 5], (tl0 + j) & 31);
        stg[j * 128 + row] = __fmul_rn(__fmul_rn(__int2float_rn(iv[j]), sr), sd);  // 0 off the edge
    }
    ptx::fence_proxy_async_smem();
    if (leader) ptx::bulk_wait_read0();  // previous group's store has read the other buffer
    if (!wg.sync(lane, P.err)) return false;
    if constexpr (EPI == EPI_F32) {  // token row >> 3 of the group; this thread's 16 channels
        const int j = row >> 3, p = row & 7;
        float m = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = *reinterpret_cast<const float4*>(stg + j * 128 + 32 * q + 4 * p);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (p == 0 && j < nv) atomicMax(&P.rowmax[ti.r0 + j0 + j], __float_as_uint(m));
    }
    if (nv == GT && P.tma_out) {
        // (a CTA pair's last tile may hold a channel block wholly beyond nout)
        if (leader && ti.mb * 128 < P.nout) {
            ptx::tma_store_2d(tmO, ti.mb * 128, ti.r0 + j0, ptx::smem_addr(stg));
            ptx::bulk_commit();
        }
    } else if (chok) {
#pragma unroll
        for (int j = 0; j < GT; ++j)
            if (j < nv) P.out_f32[(long long)(ti.r0 + j0 + j) * P.nout + col] = stg[j * 128 + row];
    }
    return true;
}

// The persistent tile loop's worker index and count: the CTA's, or for CTA
// pairs the pair's.  Read at each use: holding them (and a capturing decode
// lambda) in registers across the whole kernel measured 12% slower on the
// int8-weight GEMMs.
template <bool PAIR>
__device__ __forceinline__ int tile_worker() {
    return PAIR ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
}
template <bool PAIR>
__device__ __forceinline__ int tile_workers() {
    return PAIR ? (int)ptx::cluster_count_x() : (int)gridDim.x;
}
// a pair's tile names its 256-channel block; each CTA takes its 128
template <bool PAIR>
__device__ __forceinline__ TileInfo decode_tile(const Params& P, int tile, const TileRef& r, uint32_t rank) {
    TileInfo t = decode(P, tile, r);
    if constexpr (PAIR) t.mb = 2 * t.mb + (int)rank;
    return t;
}

template <int EPI, int BNV, bool AF16, bool PAIR = false>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const __grid_constant__ CUtensorMap tmXb,
               const __grid_constant__ CUtensorMap tmO, const Params P) {
    using TL = Tile<BNV, AF16, PAIR>;
    constexpr int BN = TL::BN, NS = TL::NS, NP = TL::NP, NAP = TL::NAB, HALF = TL::HALF, NGRP = TL::NGRP;
    constexpr int SPS = TL::SPS, CKP = CK / SPS;  // stages per step; steps per exact chunk
    constexpr int A_BYTES = TL::A_BYTES, B_BYTES = TL::B_BYTES, STAGE_BYTES = TL::STAGE_BYTES;
    constexpr int NBARS = TL::NBARS;
    constexpr uint32_t TM_A = TL::TM_A;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint8_t* stg = smem + NS * STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * STAGE_BYTES + 4 * STG_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA pairs: this CTA's rank in its pair (0 issues the MMAs); tiles go to
    // pairs, the pair's index and count (tile_worker / tile_workers) replacing
    // the CTA's
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;

    auto bar = [&](int i) { return ptx::smem_addr(bars + i); };
    auto fullp = [&](int sp) { return bar(sp); };        // the stages of step slot sp loaded
    auto emptyp = [&](int sp) { return bar(NP + sp); };  // step slot sp consumed by the MMAs
    auto afull = [&](int p) { return bar(2 * NP + p); };  // A-slot pair p converted
    auto accfull = [&](int b) { return bar(2 * NP + NAP + b); };
    auto accempty = [&](int b) { return bar(2 * NP + NAP + 2 + b); };
    const uint32_t done_bar = bar(2 * NP + NAP + 4);
    auto wg_bar = [&](int h) { return bar(2 * NP + NAP + 5 + h); };

    if (threadIdx.x == 0) {
        for (int sp = 0; sp < NP; ++sp) {
            ptx::mbar_init(fullp(sp), 1);
            ptx::mbar_init(emptyp(sp), 1);
        }
        for (int p = 0; p < NAP; ++p) ptx::mbar_init(afull(p), 4);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull(b), 1);
            ptx::mbar_init(accempty(b), PAIR ? 16 : 8);  // pairs: both CTAs' drain warps
        }
        ptx::mbar_init(done_bar, 1);
        ptx::mbar_init(wg_bar(0), 4);
        ptx::mbar_init(wg_bar(1), 4);
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmW);
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmXb);
        if (EPI != EPI_BF16MSG) ptx::prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), TM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // the peer's barriers exist before any remote arrival
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int total_tiles = P.tile_prefix[P.G] * P.mb_count;
    // K stages in steps of SPS; with pairs, an odd count gets one more stage
    // entirely beyond K, which TMA fills with zeros (it adds nothing to the sums)
    const int KSP = (P.K / BK + SPS - 1) / SPS;
    const int nchunks = (KSP + CKP - 1) / CKP;
    const int wgi = warp >> 2;

    if (wgi == 0) {
        reg_dealloc<REG_CTRL>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------- TMA producer
            // One pair of stages per step: one wait for the pair slot, one
            // expect_tx for both stages' bytes, then the loads of both.
            uint32_t pr = 0;  // stage pairs issued
            bool ok = true;
            TileRef e_next = tile_entry(P, tile_worker<PAIR>(), total_tiles);
            for (int tile = tile_worker<PAIR>(); ok && tile < total_tiles; tile += tile_workers<PAIR>()) {
                const TileInfo ti = decode_tile<PAIR>(P, tile, e_next, rank);
                e_next = tile_entry(P, tile + tile_workers<PAIR>(), total_tiles);
                const int yw0 = ti.set * P.rows_per_set + ti.mb * 128;
                const int yw1 = yw0 + P.box1_off;
                // nearly full tiles take their activations in one box of all
                // the CTA's rows (same shared-memory image as the 32-row
                // boxes), ragged ones only the 32-row boxes they need; in a
                // pair each CTA takes one half of the MMA's N (the even CTA
                // the first)
                const int brows = PAIR ? ti.nmma / 2 : ti.nmma;
                const int brow0 = PAIR ? ti.r0 + (int)rank * brows : ti.r0;
                const int nb = (brows + BOX_ROWS - 1) / BOX_ROWS;
                const bool one_box = nb == (PAIR ? BN / 2 : BN) / BOX_ROWS;
                const uint32_t bytes = SPS * (A_BYTES + nb * BOX_BYTES);
                for (int kp = 0; kp < KSP; ++kp, ++pr) {
                    const int sp = pr % NP;
                    if (!ptx::mbar_wait(emptyp(sp), ((pr / NP) & 1) ^ 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    if constexpr (PAIR) {
                        // both CTAs' loads complete on the even CTA's barrier,
                        // whose producer alone expects the bytes of both (the
                        // same count: both take the same boxes).  The odd
                        // CTA's bytes may land before that arrival; the phase
                        // cannot complete without it, and the odd CTA cannot
                        // load the slot again before the MMAs of this phase
                        // released it.
                        const uint32_t fb = ptx::mapa(fullp(sp), 0);
                        if (rank == 0) ptx::mbar_expect_tx(fullp(sp), 2 * bytes);
#pragma unroll
                        for (int j = 0; j < SPS; ++j) {
                            const uint32_t st = ptx::smem_addr(stages + (SPS * sp + j) * STAGE_BYTES);
                            const int x = (SPS * kp + j) * BK;  // beyond K (padding stage): zero fill
                            ptx::tma_load_2d_pair(st + B_BYTES, &tmW, x, yw0, fb);
                            if (one_box) {
                                ptx::tma_load_2d_pair(st, &tmXb, x, brow0, fb);
                            } else {
                                for (int b = 0; b < nb; ++b)
                                    ptx::tma_load_2d_pair(st + b * BOX_BYTES, &tmX, x, brow0 + b * BOX_ROWS, fb);
                            }
                        }
                    } else {
                        ptx::mbar_expect_tx(fullp(sp), bytes);
#pragma unroll
                        for (int j = 0; j < SPS; ++j) {
                            const uint32_t st = ptx::smem_addr(stages + (SPS * sp + j) * STAGE_BYTES);
                            const int x = (SPS * kp + j) * BK;  // beyond K (padding stage): zero fill
                            if constexpr (AF16) {  // one 128-row fp16 box, 128B swizzle
                                ptx::tma_load_2d(st + B_BYTES, &tmW, x, yw0, fullp(sp));
                            } else {               // two 64-row int8 boxes, 64B swizzle
                                ptx::tma_load_2d(st + B_BYTES, &tmW, x, yw0, fullp(sp));
                                ptx::tma_load_2d(st + B_BYTES + 4096, &tmW, x, yw1, fullp(sp));
                            }
                            if (one_box) {
                                ptx::tma_load_2d(st, &tmXb, x, ti.r0, fullp(sp));
                            } else {
                                for (int b = 0; b < nb; ++b)
                                    ptx::tma_load_2d(st + b * BOX_BYTES, &tmX, x, ti.r0 + b * BOX_ROWS, fullp(sp));
                            }
                        }
                    }
                }
            }
            if (!ok) {  // let the loads already issued land before leaving
                if (!PAIR || rank == 0) {
                    for (uint32_t j = (pr > NP ? pr - NP : 0); j < pr; ++j)
                        mbar_wait_quiet(fullp(j % NP), (j / NP) & 1, DRAIN_NS);
                } else {  // the odd CTA's loads count on the even CTA's barriers
                    const uint64_t t0 = ptx::globaltimer();
                    while (ptx::globaltimer() - t0 < DRAIN_NS) __nanosleep(1000);
                }
            }
        } else if (warp == 1 && lane == 0 && (!PAIR || rank == 0)) {
            // --------------------------------------------- MMA issuer
            // (pairs: the even CTA issues the pair's M = 256 MMAs)
            // Per step: one wait (int8 weights: for the converted weights of
            // the stage pair, which the converter signals only after it has
            // seen the pair's loads land; fp16 weights: for the stage's loads),
            // 8 or 4 MMAs at constant descriptor offsets, one commit that
            // releases the step's slot.
            uint32_t pr = 0, q = 0;
            bool ok = true;
            const uint64_t bdesc0 = ptx::sdesc_k_sw128(ptx::smem_addr(stages));
            const uint64_t adesc0 = ptx::sdesc_k_sw128(ptx::smem_addr(stages + B_BYTES));
            TileRef e_next = tile_entry(P, tile_worker<PAIR>(), total_tiles);
            for (int tile = tile_worker<PAIR>(); ok && tile < total_tiles; tile += tile_workers<PAIR>()) {
                const TileInfo ti = decode_tile<PAIR>(P, tile, e_next, rank);
                e_next = tile_entry(P, tile + tile_workers<PAIR>(), total_tiles);
                const uint32_t idesc = ptx::idesc_f16_f32(PAIR ? 256 : 128, ti.nmma);
                for (int kp = 0; kp < KSP; ++kp, ++pr) {
                    const bool first = (kp % CKP) == 0;
                    const bool last = (kp % CKP) == CKP - 1 || kp == KSP - 1;
                    const uint32_t b = q & 1;
                    if (first) {
                        // the drains must have taken this buffer's previous chunk
                        if (!ptx::mbar_wait(accempty(b), ((q >> 1) & 1) ^ 1, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                    }
                    const int sp = pr % NP;
                    const uint32_t ready = AF16 ? fullp(sp) : afull(pr % NAP);
                    const uint32_t ready_par = AF16 ? (pr / NP) & 1 : (pr / NAP) & 1;
                    if (!ptx::mbar_wait(ready, ready_par, P.err, WAIT_NS, MOE_ERR_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>((SPS * sp * STAGE_BYTES) >> 4);
                    const uint64_t bd = bdesc0 + soff;
                    const uint32_t d = tmem + TM_ACC + b * BN;
                    if constexpr (AF16) {
                        // the A and B images have the same layout: one K step
                        // (16 elements, 32 bytes) is +2 in both descriptors
                        const uint64_t ad = adesc0 + soff;
#pragma unroll
                        for (int kk = 0; kk < SPS * BK / 16; ++kk) {
                            const uint64_t o = (kk >> 2) * (STAGE_BYTES >> 4) + (kk & 3) * 2;
                            const uint32_t acc = (kk > 0 || !first) ? 1u : 0u;
                            if constexpr (PAIR) ptx::mma_f16_ss_pair(d, ad + o, bd + o, idesc, acc);
                            else ptx::mma_f16_ss(d, ad + o, bd + o, idesc, acc);
                        }
                    } else {
                        const uint32_t abase = tmem + TM_A + (pr % NAP) * 64;
                        ptx::mma_f16_ts(d, abase, bd, idesc, first ? 0u : 1u);
#pragma unroll
                        for (int kk = 1; kk < SPS * BK / 16; ++kk)
                            ptx::mma_f16_ts(d, abase + kk * 8,
                                            bd + (kk >> 2) * (STAGE_BYTES >> 4) + (kk & 3) * 2, idesc, 1u);
                    }
                    // the step's stages (and A slots) are consumed; pairs: in both CTAs
                    if constexpr (PAIR) ptx::tc_commit_pair(emptyp(sp), 3);
                    else ptx::tc_commit(emptyp(sp));
                    if (last) {
                        if constexpr (PAIR) ptx::tc_commit_pair(accfull(b), 3);
                        else ptx::tc_commit(accfull(b));
                        ++q;
                    }
                }
            }
            // every MMA issued above must be complete before TMEM is freed
            if constexpr (PAIR) ptx::tc_commit_pair(done_bar, 1);
            else ptx::tc_commit(done_bar);
            mbar_wait_quiet(done_bar, 0, WAIT_NS);
        }
    } else if (wgi == 1 && AF16) {
        reg_dealloc<REG_IDLE>();  // fp16 weights: nothing to convert
    } else if (wgi == 1) {
        // ------------------------------------------------------- converter
        reg_dealloc<REG_CONV>();
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        // TMEM lane `row` takes weight row `row` of the tile (two 64-row boxes)
        const uint8_t* arow_base = stages + B_BYTES + (row >> 6) * 4096 + (row & 63) * 64;
        const int sw = (row >> 1) & 3;
        uint32_t pr = 0;
        bool ok = true;
        for (int tile = tile_worker<PAIR>(); ok && tile < total_tiles; tile += tile_workers<PAIR>()) {
            for (int kp = 0; kp < KSP; ++kp, ++pr) {
                const int sp = pr % NP;
                // The A slots of pair pr were last read by the MMAs of pair
                // pr - NAP, whose commit completed the `empty` phase of its
                // shared-memory slot.  With as many A pairs as shared-memory
                // pairs that phase also let the producer load pair pr, so
                // the data wait covers it.
                const uint32_t pq = pr - NAP;
                if (!warp_wait(fullp(sp), (pr / NP) & 1, P.err) ||
                    (NAP < NP && pr >= NAP && !warp_wait(emptyp(pq % NP), (pq / NP) & 1, P.err))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
                    // this thread's weight row: 64 int8 in 64-byte rows, 64B swizzle
                    const uint8_t* arow = arow_base + (2 * sp + j) * STAGE_BYTES;
                    uint4 w[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(arow + ((c ^ sw) << 4));
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        s8x4_to_f16x4(w[c].x, v[8 * c + 0], v[8 * c + 1]);
                        s8x4_to_f16x4(w[c].y, v[8 * c + 2], v[8 * c + 3]);
                        s8x4_to_f16x4(w[c].z, v[8 * c + 4], v[8 * c + 5]);
                        s8x4_to_f16x4(w[c].w, v[8 * c + 6], v[8 * c + 7]);
                    }
                    ptx::tmem_st32(tmem + lane_base + TM_A + (pr % NAP) * 64 + j * 32, v);
                    ptx::tmem_wait_st();
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(afull(pr % NAP));
            }
        }
    } else {
        // ---------------------------- chunk drain and epilogue (2 groups)
        reg_alloc<AF16 ? REG_DRAIN_F16 : REG_DRAIN>();
        const int h = wgi - 2;                 // token columns [h*HALF, h*HALF + HALF)
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const bool leader = (wq == 0) && (lane == 0);
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        uint8_t* my_stg = stg + h * 2 * STG_BYTES;
        uint32_t ngrp_done = 0;                // staged groups so far (buffer = parity)
        int rs[NGRP * GT];                     // int32 running sums of this group's columns
        uint32_t q = 0;
        bool ok = true;
        WgBarrier wgb{wg_bar(h), 0};
        TileRef e_next = tile_entry(P, tile_worker<PAIR>(), total_tiles);
        for (int tile = tile_worker<PAIR>(); ok && tile < total_tiles; tile += tile_workers<PAIR>()) {
            const TileInfo ti = decode_tile<PAIR>(P, tile, e_next, rank);
            e_next = tile_entry(P, tile + tile_workers<PAIR>(), total_tiles);
            const int tok0 = h * HALF;
            const int ng = max(0, min(NGRP, (ti.nmma - tok0 + GT - 1) / GT));
            // the staged epilogue's scales, loaded while the tile's chunks run
            constexpr int NQ = HALF / 32;
            float srv[NQ];
            float sdv = 0.f;
            if constexpr (EPI == EPI_GU || EPI == EPI_F32) {
#pragma unroll
                for (int qq = 0; qq < NQ; ++qq) {
                    const int t = tok0 + 32 * qq + lane;
                    srv[qq] = t < ti.nvalid ? P.s_row[ti.r0 + t] : 0.f;
                }
                const int col = ti.mb * 128 + row;
                sdv = col < P.nout ? P.s_ch[(long long)ti.set * P.rows_per_set + col] : 0.f;
            }
            for (int c = 0; ok && c < nchunks; ++c) {
                const uint32_t b = q & 1;
                if (!warp_wait(accfull(b), (q >> 1) & 1, P.err)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t accb = tmem + lane_base + TM_ACC + b * BN + tok0;
#pragma unroll
                for (int gi = 0; gi < NGRP; ++gi) {
                    if (gi < ng) {
                        uint32_t v[GT];
                        ptx::tmem_ld16(accb + gi * GT, v);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < GT; ++j) {
                            const int x = __float2int_rn(__uint_as_float(v[j]));
                            int& r = rs[gi * GT + j];
                            r = (c > 0) ? r + x : x;
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {  // buffer free for the MMA (pairs: the even CTA's barrier)
                    if constexpr (PAIR) ptx::mbar_arrive_cluster(ptx::mapa(accempty(b), 0));
                    else ptx::mbar_arrive(accempty(b));
                }
                ++q;
                if (c == nchunks - 1) {
                    // epilogue from the final sums, overlapping the next chunks' MMAs
                    if constexpr (EPI == EPI_GU || EPI == EPI_F32) {
                        // unrolled over the groups, so that each group's sums are a
                        // fixed slice of rs (no selection of registers per group)
#pragma unroll
                        for (int gi = 0; gi < NGRP; ++gi) {
                            if (ok && gi < ng) {
                                const int (&iv)[GT] = *reinterpret_cast<const int(*)[GT]>(&rs[gi * GT]);
                                float* buf = reinterpret_cast<float*>(my_stg + (ngrp_done & 1) * STG_BYTES);
                                if (!epilogue_staged<EPI, NQ>(P, ti, row, lane, tok0 + gi * GT, gi * GT, iv, srv,
                                                              sdv, buf, &tmO, wgb, leader))
                                    ok = false;
                                ++ngrp_done;
                            }
                        }
                    } else {
#pragma unroll 1
                        for (int gi = 0; gi < ng; ++gi) {
                            if (ok) {
                                int iv[GT];  // this group's sums (predicated moves keep rs in registers)
#pragma unroll
                                for (int g2 = 0; g2 < NGRP; ++g2)
                                    if (g2 == gi) {
#pragma unroll
                                        for (int j = 0; j < GT; ++j) iv[j] = rs[g2 * GT + j];
                                    }
                                const int j0 = tok0 + gi * GT;
                                if (EPI == EPI_I32 && P.tma_out && j0 + GT <= ti.nvalid) {
                                    if (!epilogue_tma<EPI>(P, ti, row, lane, j0, iv, my_stg, &tmO, wgb, leader))
                                        ok = false;
                                } else {
                                    epilogue_direct<EPI>(P, ti, row, lane, j0, iv);
                                }
                            }
                        }
                    }
                }
            }
        }
        if (leader) ptx::bulk_wait0();  // every tensor store has landed
    }

    // ------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    // pairs: the even CTA's MMAs (which read this CTA's shared memory and
    // write its tensor memory) have completed, and no remote arrival is due
    if constexpr (PAIR) ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, TM_COLS);
        else ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

// ------------------------------------------------------------ helpers
// Gather rows (optionally through row_index) of an int8 matrix and convert
// them to fp16 (exact); optionally copy the dispatch scale of each row.
// A row-list entry outside [0, a_rows) gives a zero row (and scale) and
// posts MOE_ERR_INDEX.
__global__ void __launch_bounds__(128)
assemble_kernel(int K, const int32_t* __restrict__ row_index, long long a_rows,
                const int8_t* __restrict__ A, long long lda, const moe_dispatch_meta* __restrict__ meta,
                __half* __restrict__ out, float* __restrict__ s_row, int* __restrict__ err) {
    const int r = blockIdx.x;
    const long long g = row_index ? row_index[r] : r;
    uint4* dst = reinterpret_cast<uint4*>(out + (long long)r * K);
    const int nch = K / 16;
    if (g < 0 || g >= a_rows) {
        for (int c = threadIdx.x; c < 2 * nch; c += blockDim.x) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        if (threadIdx.x == 0) {
            post_status(err, MOE_ERR_INDEX);
            if (meta) s_row[r] = 0.f;
        }
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(A + g * lda);
    // four 16-byte loads of the row in flight per thread before converting
    for (int c0 = threadIdx.x; c0 < nch; c0 += 4 * blockDim.x) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * blockDim.x;
            if (c < nch) w[u] = __ldg(src + c);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * blockDim.x;
            if (c < nch) {
                uint4 o0, o1;
                s8x4_to_f16x4(w[u].x, o0.x, o0.y);
                s8x4_to_f16x4(w[u].y, o0.z, o0.w);
                s8x4_to_f16x4(w[u].z, o1.x, o1.y);
                s8x4_to_f16x4(w[u].w, o1.z, o1.w);
                dst[2 * c] = o0;
                dst[2 * c + 1] = o1;
            }
        }
    }
    if (meta && threadIdx.x == 0) s_row[r] = meta[g].scale;
}

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

// The row kernels below take 16 consecutive values per thread and chunk.
// requant runs with row_threads(I) threads, enough that a row is loaded in
// one pass of two chunks per thread (I = 2048: 64 threads), so a block waits
// for memory once; retquant issues the loads of two chunks (eight 16-byte
// loads) before quantising and keeps kRowThreads (at H = 7168, 224-thread
// blocks that load a row in one pass measured slower: 643 -> 722 us).
constexpr int kRowThreads = 128;
constexpr int kRowMaxThreads = 256;
inline int row_threads(int n) {
    const int half = (n / 16 + 1) / 2;  // chunks of 16 values per thread pair
    return std::min(kRowMaxThreads, std::max(32, (half + 31) / 32 * 32));
}

__device__ __forceinline__ void load_chunk16(const float4* __restrict__ src, int c, int nch,
                                             float4 (&v)[4]) {
    if (c < nch) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(src + 4 * c + i);
    }
}

// SwiGLU and the token-wise requantisation of its output, one expert row per
// block: h = SiLU(g) * u from the gate/up GEMM's g and u (h rounded once,
// SiLU by silu_fast: the exp specification and a correctly rounded
// quotient), the row's |h| maximum, s_h = max / 127 and the codes of h as
// exact fp16 integers.  Each thread holds up to CH chunks of 16 values in
// registers (row_threads(I) threads: CH = 2 covers I <= 8192, 4 covers the
// largest I), so g and u are read once.
template <int CH>
__global__ void __launch_bounds__(kRowMaxThreads)
requant_kernel(int I, const float* __restrict__ gu, __half* __restrict__ hq, float* __restrict__ sh,
               unsigned* __restrict__ ymax) {
    __shared__ float s_red[kRowMaxThreads / 32];
    const int r = blockIdx.x;
    if (threadIdx.x == 0) ymax[r] = 0u;  // the down epilogue's row maximum of y starts at 0
    const int nch = I / 16;
    const int nt = blockDim.x;
    const float4* gsrc = reinterpret_cast<const float4*>(gu + (long long)r * 2 * I);
    const float4* usrc = gsrc + I / 4;
    float hv[CH][16];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = threadIdx.x + u * nt;
        if (c < nch) {
            float4 g4[4], u4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                g4[i] = __ldg(gsrc + 4 * c + i);
                u4[i] = __ldg(usrc + 4 * c + i);
            }
            const float gg[16] = {g4[0].x, g4[0].y, g4[0].z, g4[0].w, g4[1].x, g4[1].y, g4[1].z, g4[1].w,
                                  g4[2].x, g4[2].y, g4[2].z, g4[2].w, g4[3].x, g4[3].y, g4[3].z, g4[3].w};
            const float uu[16] = {u4[0].x, u4[0].y, u4[0].z, u4[0].w, u4[1].x, u4[1].y, u4[1].z, u4[1].w,
                                  u4[2].x, u4[2].y, u4[2].z, u4[2].w, u4[3].x, u4[3].y, u4[3].z, u4[3].w};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                hv[u][e] = __fmul_rn(silu_fast(gg[e]), uu[e]);
                amax = fmaxf(amax, fabsf(hv[u][e]));
            }
        }
    }
    // row maximum over the block
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    float m = s_red[0];
    for (int i = 1; i < nt / 32; ++i) m = fmaxf(m, s_red[i]);
    const float s = row_scale(m);
    const float rs = quant_rcp(s);
    uint4* dst = reinterpret_cast<uint4*>(hq + (long long)r * I);
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = threadIdx.x + u * nt;
        if (c < nch) {
            int q[16];
            if (s != 0.f) {
                quant_row_n<16>(hv[u], s, rs, q);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) q[e] = 0;
            }
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = codes_to_f16x2(q[2 * i], q[2 * i + 1]);
            dst[2 * c] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[2 * c + 1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
    if (threadIdx.x == 0) sh[r] = s;
}

// INT8 return message of expert row r: token-wise codes of y (its row absmax
// was reduced by the down GEMM's epilogue) into the combine row (t, j), and
// its scale.  Returns t * k + j, or -1 (and MOE_ERR_INDEX) if the row's
// dispatch slot or metadata is out of range.  Called by all threads of a
// block of kRowThreads with the same r.
__device__ __forceinline__ long long quantise_return_row(
    int r, int H, int k, int lb, int S, long long nslots, long long crow, const float* __restrict__ y,
    const unsigned* __restrict__ rowmax, const int32_t* __restrict__ expert_rows,
    const moe_dispatch_meta* __restrict__ meta, unsigned char* __restrict__ cbuf,
    float* __restrict__ cscale, int* __restrict__ err) {
    const long long g = expert_rows[r];
    if (g < 0 || g >= nslots || !meta_in_range(meta[g], S, lb, k)) {  // caller data out of range
        if (threadIdx.x == 0) post_status(err, MOE_ERR_INDEX);
        return -1;
    }
    const int nch = H / 16;
    const float4* src = reinterpret_cast<const float4*>(y + (long long)r * H);
    const int nt = blockDim.x;
    long long tj = 0;
    for (int c0 = threadIdx.x; c0 < nch; c0 += 2 * nt) {
        float4 v[2][4];
        load_chunk16(src, c0, nch, v[0]);
        load_chunk16(src, c0 + nt, nch, v[1]);
        const moe_dispatch_meta m = meta[g];
        tj = ((long long)m.src_rank * lb + m.batch_slot) * k + m.route_slot;
        uint4* dst = reinterpret_cast<uint4*>(cbuf + tj * crow);
        const float s = row_scale(__uint_as_float(rowmax[r]));
        const float rs = quant_rcp(s);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c = c0 + u * nt;
            if (c >= nch) break;
            const float x[16] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y,
                                 v[u][1].z, v[u][1].w, v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w,
                                 v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
            int q[16];
            if (s != 0.f) {
                quant_row_n<16>(x, s, rs, q);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) q[e] = 0;
            }
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = (uint32_t)(q[4 * i] & 0xff) | ((uint32_t)(q[4 * i + 1] & 0xff) << 8) |
                       ((uint32_t)(q[4 * i + 2] & 0xff) << 16) | ((uint32_t)(q[4 * i + 3] & 0xff) << 24);
            dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    const moe_dispatch_meta m = meta[g];
    tj = ((long long)m.src_rank * lb + m.batch_slot) * k + m.route_slot;
    if (threadIdx.x == 0) cscale[tj] = row_scale(__uint_as_float(rowmax[r]));
    return tj;
}

// INT8 return messages, one block per expert row.
__global__ void __launch_bounds__(kRowThreads)
retquant_kernel(int H, int k, int lb, int S, long long nslots, long long crow,
                const float* __restrict__ y, const unsigned* __restrict__ rowmax,
                const int32_t* __restrict__ expert_rows, const moe_dispatch_meta* __restrict__ meta,
                unsigned char* __restrict__ cbuf, float* __restrict__ cscale, int* __restrict__ err) {
    quantise_return_row(blockIdx.x, H, k, lb, S, nslots, crow, y, rowmax, expert_rows, meta, cbuf,
                        cscale, err);
}

// Acquire load of a readiness counter (device scope).
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *ctr >= target: gives up (false) after limit_ns of
// %globaltimer time, posting MOE_ERR_TIMEOUT, or at once when another thread
// has posted any error.  Never traps.
__device__ __forceinline__ bool wait_count(const int* ctr, int target, int* err, uint64_t limit_ns) {
    if (ld_acquire(ctr) >= target) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(64);
        if (ld_acquire(ctr) >= target) return true;
        if ((it & 7) == 0) {
            if (*reinterpret_cast<volatile int*>(err) != 0) return false;
            if (ptx::globaltimer() - t0 > limit_ns) {
                atomicCAS(err, 0, MOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// FusedCombine folded into the return messages, as the pages' fused path runs
// it ("CloudMatrix384 LLM Serving", "EP320" fused_moe listing: the combine of a
// token waits until all k contributions are in; "xDeepServe", COMBINE
// procedure).  One persistent kernel (cooperative launch, every block
// resident) takes work items from an atomic ticket: items 0 .. M-1 are the
// expert rows, M .. M+T-1 the tokens.
//   row r:    write its INT8 return message (quantise_return_row), fence,
//             then count it in ready[t];
//   token t:  one thread waits until ready[t] reaches `expected` (wait_count,
//             bounded), then the block sums the k messages as the combine
//             kernel does and writes out[t].
// Every row item is taken before any token item, by a running block that
// waits for nothing, so each wait ends once the rows are written; the bound
// only catches a count that can never be reached (a lost message, or an
// `expected` other than k), which posts MOE_ERR_TIMEOUT and skips the token.
struct RetCombine {
    int H, k, lb, S, expected;
    long long M, T, nslots, crow;
    uint64_t wait_ns;
    const float* y;
    const unsigned* rowmax;
    const int32_t* expert_rows;
    const moe_dispatch_meta* meta;
    unsigned char* cbuf;
    float* cscale;
    const float* topk_w;
    int* ready;  // [T] readiness counters, then the work ticket
    uint16_t* out;
    int* err;
};

__global__ void __launch_bounds__(kRowThreads) retcombine_kernel(const RetCombine P) {
    constexpr int kMaxK = 32;
    constexpr int kUnroll = 8;
    __shared__ long long s_item;
    __shared__ int s_ok;
    __shared__ float s_w[kMaxK], s_s[kMaxK];
    int* ticket = P.ready + P.T;
    for (;;) {
        if (threadIdx.x == 0) s_item = atomicAdd(ticket, 1);
        __syncthreads();
        const long long item = s_item;
        __syncthreads();
        if (item >= P.M + P.T) return;
        if (item < P.M) {
            const long long tj = quantise_return_row((int)item, P.H, P.k, P.lb, P.S, P.nslots, P.crow,
                                                     P.y, P.rowmax, P.expert_rows, P.meta, P.cbuf,
                                                     P.cscale, P.err);
            if (tj < 0) continue;
            __threadfence();  // this thread's message stores, device-wide, before the count
            __syncthreads();
            if (threadIdx.x == 0) atomicAdd(P.ready + tj / P.k, 1);
            continue;
        }
        const long long t = item - P.M;
        if (threadIdx.x == 0) s_ok = wait_count(P.ready + t, P.expected, P.err, P.wait_ns);
        __syncthreads();
        if (!s_ok) continue;
        __threadfence();  // the k messages are visible from here on
        if (threadIdx.x < P.k) {
            s_w[threadIdx.x] = P.topk_w[t * P.k + threadIdx.x];
            s_s[threadIdx.x] = __ldcg(P.cscale + t * P.k + threadIdx.x);
        }
        __syncthreads();
        const int k = P.k;
        const unsigned char* rows = P.cbuf + t * k * P.crow;
        uint4* orow = reinterpret_cast<uint4*>(P.out + t * P.H);
        for (int c = threadIdx.x; c < P.H / 16; c += kRowThreads) {
            uint4 q[kUnroll][2];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j)
                if (j < k) load16<true, true>(rows + j * P.crow, c, q[j]);
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
            for (int j = 0; j < kUnroll; ++j)
                if (j < k) accumulate16<true>(q[j], s_w[j], s_s[j], acc);
            for (int j = kUnroll; j < k; ++j) {
                uint4 q2[2];
                load16<true, true>(rows + j * P.crow, c, q2);
                accumulate16<true>(q2, s_w[j], s_s[j], acc);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 o;
                o.x = pack_bf16x2(acc[8 * h + 0], acc[8 * h + 1]);
                o.y = pack_bf16x2(acc[8 * h + 2], acc[8 * h + 3]);
                o.z = pack_bf16x2(acc[8 * h + 4], acc[8 * h + 5]);
                o.w = pack_bf16x2(acc[8 * h + 6], acc[8 * h + 7]);
                orow[2 * c + h] = o;
            }
        }
        __syncthreads();  // s_w / s_s are free for the next token
    }
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

// Persistent grid: one CTA per SM, or, for CTA pairs, as many two-CTA
// clusters as the device holds at once (a GPC with an odd number of SMs
// leaves one out).  The clusters never wait on one another.
template <int EPI, int BNV, bool AF16 = false, bool PAIR = false>
cudaError_t launch_gemm(const Params& P, const CUtensorMap& w, const CUtensorMap (&x)[2],
                        const CUtensorMap& o, cudaStream_t st) {
    constexpr int smem = Tile<BNV, AF16, PAIR>::SMEM_BYTES;
    auto* kern = gemm_tc_kernel<EPI, BNV, AF16, PAIR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int slot = EPI == EPI_GU ? 0 : 1;
    if constexpr (PAIR) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        static int clusters[64][4] = {};  // per device and kernel form
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64) dev = 0;
        int& nc = clusters[dev][EPI];
        if (!nc) {
            int n = 0;
            if ((e = cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg)) != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
            nc = std::min(n, sm_count() / 2);
        }
        cfg.gridDim = dim3((unsigned)(2 * nc));
        if (cudaEvent_t ev = prof_event(slot, 0)) cudaEventRecord(ev, st);
        e = cudaLaunchKernelEx(&cfg, kern, w, x[0], x[1], o, P);
        if (cudaEvent_t ev = prof_event(slot, 1)) cudaEventRecord(ev, st);
        count_launches(1);
        return e != cudaSuccess ? e : cudaGetLastError();
    } else {
        if (cudaEvent_t ev = prof_event(slot, 0)) cudaEventRecord(ev, st);
        kern<<<sm_count(), THREADS, smem, st>>>(w, x[0], x[1], o, P);
        if (cudaEvent_t ev = prof_event(slot, 1)) cudaEventRecord(ev, st);
        count_launches(1);
        return cudaGetLastError();
    }
}

bool weight_map(CUtensorMap* m, const int8_t* w, int K, uint64_t rows) {
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, K, rows, BK, 64, CU_TENSOR_MAP_SWIZZLE_64B);
}

// fp16 copy of the weights: boxes of 64 K x 128 rows, the same 128B-swizzled
// K-major image as the activations.
bool weight_map(CUtensorMap* m, const uint16_t* w, int K, uint64_t rows) {
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w, K, rows, BK, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Activation maps: [0] boxes of BOX_ROWS rows, [1] boxes of bn rows (a tile).
bool act_map(CUtensorMap (&m)[2], const __half* x, int K, uint64_t rows, int bn) {
    return make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, rows, BK, BOX_ROWS,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, rows, BK, (uint32_t)bn,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output map of the epilogue's tensor stores: [rows][cols] 32-bit elements,
// boxes of box_cols x GT rows, no swizzle.
bool out_map(CUtensorMap* m, const void* base, bool is_int, uint64_t cols, uint64_t rows,
             uint32_t box_cols) {
    return make_map(m, is_int ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                    base, cols, rows, box_cols, GT, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace tc

// Exact grouped int8 GEMM with int32 output on the tensor-core path.
// Workspace: [status 256 B][tile prefix][fp16 copy of the A rows].
cudaError_t launch_grouped_gemm_tc(int n_groups, const int32_t* offsets, long long max_rows,
                                   const int32_t* row_index, const int8_t* A, long long lda,
                                   const int8_t* B, int N, int K, int32_t* C, void* ws,
                                   cudaStream_t st) {
    using namespace tc;
    const GemmWs gw = gemm_ws(n_groups, max_rows, K);
    int* err = ws_ptr<int>(ws, 0);
    int32_t* tp = ws_ptr<int32_t>(ws, gw.tiles);
    int4* ttab = ws_ptr<int4>(ws, gw.ttab);
    __half* a16 = ws_ptr<__half>(ws, gw.a16);
    cudaError_t e = clear_status(ws, st);
    if (e != cudaSuccess) return e;
    if ((e = launch_tile_prefix(n_groups, BN_LARGE, offsets, max_rows, n_groups, tp, err, st, ttab)) !=
        cudaSuccess)
        return e;
    // the rows of A are the caller's: no bound on the row list's entries here
    assemble_kernel<<<(unsigned)max_rows, 128, 0, st>>>(K, row_index, LLONG_MAX, A, lda, nullptr, a16,
                                                        nullptr, err);
    count_launches(1);
    CUtensorMap mw, mx[2], mo;
    const bool tma_out = N % 128 == 0;
    if (!weight_map(&mw, B, K, (uint64_t)n_groups * N) || !act_map(mx, a16, K, (uint64_t)max_rows, BN_LARGE) ||
        (tma_out && !out_map(&mo, C, true, N, (uint64_t)max_rows, 128)))
        return cudaErrorInvalidValue;
    if (!tma_out) mo = mx[0];  // unused
    Params P = {};
    P.G = n_groups; P.offsets = offsets; P.tile_prefix = tp; P.ttab = ttab; P.g2s = nullptr;
    P.K = K; P.rows_per_set = N; P.nout = N; P.mb_count = (N + 127) / 128; P.box1_off = 64;
    P.c_i32 = C; P.err = err; P.tma_out = tma_out;
    return launch_gemm<EPI_I32, BN_LARGE>(P, mw, mx, mo, st);
}

namespace tc {

template <int BNV, bool AF16, bool PAIR = false>
cudaError_t ffn_tc(const Dims& d, const void* dbuf, long long meta_off,
                   const int32_t* expert_offsets, const int32_t* expert_rows,
                   const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                   const WsLayout& wl, cudaStream_t st, const FusedCombine& fc, bool clear,
                   bool rows_ready) {
    const long long M = (long long)d.T * d.k;
    const moe_dispatch_meta* meta =
        reinterpret_cast<const moe_dispatch_meta*>(static_cast<const char*>(dbuf) + meta_off);
    int* err = ws_ptr<int>(ws, 0);
    int32_t* tp = ws_ptr<int32_t>(ws, wl.tiles);
    int4* ttab = ws_ptr<int4>(ws, wl.ttab);
    float* s_row = ws_ptr<float>(ws, wl.s_row);
    float* sh = ws_ptr<float>(ws, wl.sh);
    __half* a16 = ws_ptr<__half>(ws, wl.a16);
    float* gubuf = ws_ptr<float>(ws, wl.gubuf);
    unsigned* ymax = ws_ptr<unsigned>(ws, wl.rowmax);
    __half* hq16 = ws_ptr<__half>(ws, wl.hq16);
    float* ybuf = ws_ptr<float>(ws, wl.ybuf);
    unsigned char* cb = static_cast<unsigned char*>(cbuf);
    const int int8_ret = d.cfmt == MOE_MSG_INT8;
    const int E_w = w.n_sets;
    cudaError_t e;

    if (clear && (e = clear_status(ws, st)) != cudaSuccess) return e;
    const bool fuse = fc.out != nullptr && int8_ret;
    int* ready = ws_ptr<int>(ws, wl.ready);
    if (fuse) {  // readiness counters and the work ticket start at zero
        if ((e = cudaMemsetAsync(ready, 0, sizeof(int) * (d.T + 1), st)) != cudaSuccess) return e;
        count_launches(1);
    }
    // experts with few rows go to the matrix-vector kernels (same outputs),
    // listed by the tile-prefix kernel
    const int narrow = narrow_expert_rows(d);
    int32_t* nlist = narrow > 0 ? ws_ptr<int32_t>(ws, wl.narrow) : nullptr;
    if ((e = launch_tile_prefix(d.E_phys, BNV, expert_offsets, M, E_w, tp, err, st, ttab,
                                w.phys_to_weight, narrow, nlist)) != cudaSuccess)
        return e;
    if (!rows_ready) {  // else the dispatch of moe_layer wrote them (launch_dispatch, stage_rows)
        assemble_kernel<<<(unsigned)M, 128, 0, st>>>(d.H, expert_rows, d.nslots,
                                                     static_cast<const int8_t*>(dbuf), d.drow, meta, a16,
                                                     s_row, err);
        count_launches(1);
    }

    CUtensorMap mwgu, mx1[2], mo1, mwd, mx2[2], mo2;
    const bool wmaps = AF16 ? weight_map(&mwgu, w.w_gate_up_f16, d.H, (uint64_t)E_w * 2 * d.I) &&
                                  weight_map(&mwd, w.w_down_f16, d.I, (uint64_t)E_w * d.H)
                            : weight_map(&mwgu, w.w_gate_up, d.H, (uint64_t)E_w * 2 * d.I) &&
                                  weight_map(&mwd, w.w_down, d.I, (uint64_t)E_w * d.H);
    constexpr int XBOX = PAIR ? BNV / 2 : BNV;  // a CTA's token rows of a full tile
    if (!wmaps || !act_map(mx1, a16, d.H, (uint64_t)M, XBOX) ||
        !out_map(&mo1, gubuf, false, (uint64_t)2 * d.I, (uint64_t)M, 128) ||
        !act_map(mx2, hq16, d.I, (uint64_t)M, XBOX))
        return cudaErrorInvalidValue;
    const bool y_tma = int8_ret && d.H >= 128;
    if (y_tma) {
        if (!out_map(&mo2, ybuf, false, (uint64_t)d.H, (uint64_t)M, 128)) return cudaErrorInvalidValue;
    } else {
        mo2 = mo1;  // unused
    }

    constexpr int CB = PAIR ? 256 : 128;  // channels per tile
    Params P1 = {};
    P1.G = d.E_phys; P1.offsets = expert_offsets; P1.tile_prefix = tp; P1.ttab = ttab;
    P1.g2s = w.phys_to_weight;
    P1.K = d.H; P1.rows_per_set = 2 * d.I; P1.nout = 2 * d.I; P1.mb_count = (2 * d.I + CB - 1) / CB; P1.box1_off = 64;
    P1.s_row = s_row; P1.s_ch = w.s_gate_up; P1.out_f32 = gubuf; P1.err = err;
    P1.tma_out = 1;
    if ((e = launch_gemm<EPI_GU, BNV, AF16, PAIR>(P1, mwgu, mx1, mo1, st)) != cudaSuccess) return e;
    if (narrow > 0 &&
        (e = launch_gemv_gate_up(d, dbuf, meta, expert_offsets, expert_rows, w, gubuf, err, nlist, 2,
                                 st)) != cudaSuccess)
        return e;

    if ((e = launch_requant_rows(d.I, M, gubuf, hq16, sh, ymax, st)) != cudaSuccess) return e;

    Params P2 = {};
    P2.G = d.E_phys; P2.offsets = expert_offsets; P2.tile_prefix = tp; P2.ttab = ttab;
    P2.g2s = w.phys_to_weight;
    P2.K = d.I; P2.rows_per_set = d.H; P2.nout = d.H; P2.mb_count = (d.H + CB - 1) / CB; P2.box1_off = 64;
    P2.s_row = sh; P2.s_ch = w.s_down; P2.err = err; P2.tma_out = y_tma;
    if (int8_ret) {
        P2.out_f32 = ybuf; P2.rowmax = ymax;
        if ((e = launch_gemm<EPI_F32, BNV, AF16, PAIR>(P2, mwd, mx2, mo2, st)) != cudaSuccess) return e;
        if (narrow > 0 &&
            (e = launch_gemv_down(d, expert_offsets, w, hq16, sh, ybuf, ymax, err, nlist, 3, st)) !=
                cudaSuccess)
            return e;
        if (fuse) {
            RetCombine R;
            R.H = d.H; R.k = d.k; R.lb = d.lb; R.S = d.S; R.expected = fc.expected;
            R.M = M; R.T = d.T; R.nslots = d.nslots; R.crow = d.crow; R.wait_ns = fc.wait_ns;
            R.y = ybuf; R.rowmax = ymax; R.expert_rows = expert_rows; R.meta = meta; R.cbuf = cb;
            R.cscale = reinterpret_cast<float*>(cb + scale_off); R.topk_w = fc.topk_w; R.ready = ready;
            R.out = fc.out; R.err = err;
            // every block resident (cooperative launch): blocks wait on counters
            // that other blocks of this launch advance
            int per_sm = 0;
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, retcombine_kernel, kRowThreads,
                                                                   0)) != cudaSuccess)
                return e;
            const long long items = M + d.T;
            const unsigned grid = (unsigned)std::max<long long>(
                1, std::min<long long>(items, (long long)std::max(per_sm, 1) * sm_count()));
            void* args[] = {&R};
            if ((e = cudaLaunchCooperativeKernel((const void*)retcombine_kernel, dim3(grid),
                                                 dim3(kRowThreads), args, 0, st)) != cudaSuccess)
                return e;
        } else {
            retquant_kernel<<<(unsigned)M, kRowThreads, 0, st>>>(
                d.H, d.k, d.lb, d.S, d.nslots, d.crow, ybuf, ymax, expert_rows, meta, cb,
                reinterpret_cast<float*>(cb + scale_off), err);
        }
        count_launches(1);

    } else {
        P2.expert_rows = expert_rows; P2.meta = meta; P2.cbuf = cb; P2.crow = d.crow; P2.k = d.k; P2.lb = d.lb;
        P2.S = d.S; P2.nslots = d.nslots;
        if ((e = launch_gemm<EPI_BF16MSG, BNV, AF16, PAIR>(P2, mwd, mx2, mo2, st)) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace tc

// fp16 copy of an int8 array (exact): 16 values per thread and step, the
// tail of n % 16 values one per thread.
__global__ void __launch_bounds__(256) weights_to_f16_kernel(const int8_t* __restrict__ src, long long n,
                                                             uint16_t* __restrict__ dst) {
    const long long nv = n / 16;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
        const uint4 w = __ldg(s4 + i);
        uint4 o0, o1;
        s8x4_to_f16x4(w.x, o0.x, o0.y);
        s8x4_to_f16x4(w.y, o0.z, o0.w);
        s8x4_to_f16x4(w.z, o1.x, o1.y);
        s8x4_to_f16x4(w.w, o1.z, o1.w);
        d4[2 * i] = o0;
        d4[2 * i + 1] = o1;
    }
    if (blockIdx.x == 0)
        for (long long i = nv * 16 + threadIdx.x; i < n; i += blockDim.x)
            dst[i] = __half_as_ushort(__int2half_rn(src[i]));
}

cudaError_t launch_weights_to_f16(const int8_t* src, long long n, uint16_t* dst, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const long long nv = n / 16;
    const long long want = std::max<long long>(1, (nv + 255) / 256);
    const unsigned grid = (unsigned)std::min<long long>(want, 8LL * tc::sm_count());
    weights_to_f16_kernel<<<grid, 256, 0, st>>>(src, n, dst);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_requant_rows(int I, long long M, const float* gu, void* hq16, float* sh, unsigned* ymax,
                                cudaStream_t st) {
    const int nt = tc::row_threads(I);
    if (I / 16 <= 2 * nt)
        tc::requant_kernel<2><<<(unsigned)M, nt, 0, st>>>(I, gu, static_cast<__half*>(hq16), sh, ymax);
    else
        tc::requant_kernel<4><<<(unsigned)M, nt, 0, st>>>(I, gu, static_cast<__half*>(hq16), sh, ymax);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_retquant_rows(const Dims& d, long long M, const float* y, const unsigned* rowmax,
                                 const int32_t* expert_rows, const moe_dispatch_meta* meta,
                                 unsigned char* cbuf, float* cscale, int* err, cudaStream_t st) {
    tc::retquant_kernel<<<(unsigned)M, tc::kRowThreads, 0, st>>>(
        d.H, d.k, d.lb, d.S, d.nslots, d.crow, y, rowmax, expert_rows, meta, cbuf, cscale, err);
    count_launches(1);
    return cudaGetLastError();
}

// Decode-sized batches (at most 32 routed rows per expert on average) take
// 64-token tiles on the int8 weights: their tiles are mostly weight
// streaming, and the smaller activation region doubles the stages in flight.
// Larger batches take the fp16 weight copies when the caller gives them
// (256-token tiles, nothing converted on the SM), else 192-token tiles on the
// int8 weights.
cudaError_t launch_ffn_tc(const Dims& d, const void* dbuf, long long meta_off,
                          const int32_t* expert_offsets, const int32_t* expert_rows,
                          const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                          const WsLayout& wl, cudaStream_t st, const FusedCombine& fc, bool clear,
                          bool rows_ready) {
    const long long M = (long long)d.T * d.k;
    if (M <= 32LL * d.E_phys)
        return tc::ffn_tc<tc::BN_DECODE, false>(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf,
                                                scale_off, ws, wl, st, fc, clear, rows_ready);
    if (w.w_gate_up_f16 && w.w_down_f16)
        return tc::ffn_tc<tc::BN_F16, true, tc::kPairF16>(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf,
                                            scale_off, ws, wl, st, fc, clear, rows_ready);
    return tc::ffn_tc<tc::BN_LARGE, false>(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf,
                                           scale_off, ws, wl, st, fc, clear, rows_ready);
}

}  // namespace moe
