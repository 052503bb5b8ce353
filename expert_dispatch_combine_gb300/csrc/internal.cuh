// internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Derived sizes of one layer shape.
struct Dims {
    int T, H, E_log, E_phys, k, I, R, S;
    int lb, epr, mt;
    int dfmt, cfmt;
    long long drow;  // dispatch row bytes
    long long crow;  // combine row bytes
    long long nslots;
};

inline Dims make_dims(const moe_shape& s) {
    Dims d;
    d.T = s.T; d.H = s.H; d.E_log = s.E_log; d.E_phys = s.E_phys; d.k = s.k; d.I = s.I;
    d.R = s.n_ranks; d.S = s.n_src_ranks;
    d.lb = d.T / d.S;
    d.epr = d.E_phys / d.R;
    d.mt = d.lb * (d.k < d.epr ? d.k : d.epr);
    d.dfmt = s.dispatch_fmt; d.cfmt = s.combine_fmt;
    d.drow = (long long)d.H * (d.dfmt == MOE_MSG_INT8 ? 1 : 2);
    d.crow = (long long)d.H * (d.cfmt == MOE_MSG_INT8 ? 1 : 2);
    d.nslots = (long long)d.R * d.S * d.mt;
    return d;
}

inline long long align_up(long long v, long long a) { return (v + a - 1) / a * a; }

// The tensor-core expert FFN needs K multiples of 64 for both GEMMs.
inline bool ffn_uses_tc(const Dims& d) { return d.H % 64 == 0 && d.I % 64 == 0; }

// Token rows per tile of the tensor-core grouped GEMM.
constexpr int kTcTileRows = 192;
// Token rows per tile when the caller gives fp16 copies of the weights.
constexpr int kTcTileRowsF16 = 256;
// Token rows per tile of its decode variant (few rows per expert).
constexpr int kTcMinTileRows = 64;
// Routed rows per expert (on average) up to which the expert FFN streams the
// weights through CUDA-core matrix-vector products instead of the tensor cores.
constexpr int kGemvRowsPerExpert = 4;
// Alongside the tensor-core GEMMs, experts with at most this many routed rows
// (one pass of the matrix-vector kernels' 8 token rows, so their weights
// stream once) are computed by the matrix-vector kernels: for them the
// tensor-core pipeline is bound by converting the whole expert's weights for
// a handful of tokens.  Measured at c2_decode_zipf: 8 rows 8.77 ms per layer,
// 12 rows 8.83, 16 rows 8.84, 24 rows 9.16, 48 rows 9.60 (each extra pass
// streams the weights again).
constexpr int kNarrowExpertRows = 8;

// Token tiles of a grouped GEMM over n_groups groups and max_rows rows, at
// most bm rows per tile (each group adds at most one partial tile).
inline long long tile_table_entries(int n_groups, long long max_rows, int bm) {
    return max_rows / bm + n_groups + 1;
}

// Workspace carve-up.  Every region is 256-byte aligned; offset 0 holds the
// int32 device status word (MOE_OK or the first error a kernel posted).
struct WsLayout {
    long long slot_local;  // int32 [T*k]   slot of (t, j) within its (dst, src) pair
    long long erank;       // int32 [T*k]   rank of token t among its source's tokens for expert p
    long long hist;        // int32 [S][E_phys]
    long long src_base;    // int32 [S][E_phys]
    long long tiles;       // int32 [E_phys + 1]  grouped-GEMM tile prefix
    long long ttab;        // int4  [tile_table_entries]  (set, first row, rows, group) per token tile
    long long sh;          // f32   [T*k]   requantisation scale of h
    long long ready;       // int32 [T+1]   return messages in per token, then a work ticket (fused combine)
    long long narrow;      // int32 [E_phys+1]  number of narrow experts, then their ids
    // SIMT expert FFN
    long long acc_gu;      // int32 [T*k][2I]
    long long hq;          // int8  [T*k][I]
    long long acc_d;       // int32 [T*k][H]
    // tensor-core expert FFN
    long long rowmax;      // u32   [T*k]     absmax of y (float bits)
    long long s_row;       // f32   [T*k]     dispatch scale of each expert row
    long long a16;         // fp16  [T*k][H]  expert input rows
    long long gubuf;       // f32   [T*k][2I] gate and up projections g, u
    long long hq16;        // fp16  [T*k][I]  requantised SwiGLU output
    long long ybuf;        // f32   [T*k][H]  expert output (INT8 return messages only)
    long long total;
    bool tc;
};

inline WsLayout make_ws(const Dims& d) {
    WsLayout w = {};
    long long o = 256;
    const long long tk = (long long)d.T * d.k;
    w.slot_local = o; o = align_up(o + 4 * tk, 256);
    w.erank = o;      o = align_up(o + 4 * tk, 256);
    w.hist = o;       o = align_up(o + 4LL * d.S * d.E_phys, 256);
    w.src_base = o;   o = align_up(o + 4LL * d.S * d.E_phys, 256);
    w.tiles = o;      o = align_up(o + 4LL * (d.E_phys + 1), 256);
    w.ttab = o;       o = align_up(o + 16LL * tile_table_entries(d.E_phys, tk, kTcMinTileRows), 256);
    w.sh = o;         o = align_up(o + 4 * tk, 256);
    w.ready = o;      o = align_up(o + 4LL * (d.T + 1), 256);
    w.narrow = o;     o = align_up(o + 4LL * (d.E_phys + 1), 256);
    w.tc = ffn_uses_tc(d);
    if (w.tc) {
        w.rowmax = o; o = align_up(o + 4 * tk, 256);
        w.s_row = o;  o = align_up(o + 4 * tk, 256);
        w.a16 = o;    o = align_up(o + 2 * tk * d.H, 256);
        w.gubuf = o;  o = align_up(o + 8 * tk * d.I, 256);
        w.hq16 = o;   o = align_up(o + 2 * tk * d.I, 256);
        if (d.cfmt == MOE_MSG_INT8) { w.ybuf = o; o = align_up(o + 4 * tk * d.H, 256); }
    } else {
        w.acc_gu = o; o = align_up(o + 4 * tk * 2 * d.I, 256);
        w.hq = o;     o = align_up(o + tk * d.I, 256);
        w.acc_d = o;  o = align_up(o + 4 * tk * d.H, 256);
    }
    w.total = o;
    return w;
}

// Workspace of moe_grouped_gemm_s8: [status][tile prefix][tile table][fp16 A rows].
struct GemmWs {
    long long tiles, ttab, a16, total;
};
inline GemmWs gemm_ws(int n_groups, long long max_rows, int K) {
    GemmWs w;
    w.tiles = 256;
    w.ttab = w.tiles + align_up(4LL * (n_groups + 1), 256);
    w.a16 = w.ttab + align_up(16LL * tile_table_entries(n_groups, max_rows, kTcMinTileRows), 256);
    w.total = w.a16 + align_up(2LL * max_rows * K, 256);
    return w;
}
inline long long gemm_ws_bytes(int n_groups, long long max_rows, int K) {
    return gemm_ws(n_groups, max_rows, K).total;
}

template <typename T>
inline T* ws_ptr(void* ws, long long off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// Number of kernels (and memsets) this library has enqueued in this process.
void count_launches(int n);

#ifdef __CUDACC__
// Posts `code` to the workspace status word unless an earlier code is there
// (the first one posted stays).
__device__ __forceinline__ void post_status(int* err, int code) { atomicCAS(err, 0, code); }

// Whether a dispatch slot's metadata names a message of this shape (the
// slot may hold stale or foreign contents if a row list is corrupt).
__device__ __forceinline__ bool meta_in_range(const moe_dispatch_meta& m, int S, int lb, int k) {
    return (unsigned)m.src_rank < (unsigned)S && (unsigned)m.batch_slot < (unsigned)lb &&
           (unsigned)m.route_slot < (unsigned)k;
}
#endif

// Clears the workspace status word (one 256-byte memset) on `st`.
cudaError_t clear_status(void* ws, cudaStream_t st);
// Trampoline area of the two-hop dispatch: [T][drow] message rows, [T]
// moe_dispatch_meta (route_slot = k: the routes follow), [T][k] int32
// physical expert ids.  Trampoline s holds the rows of source rank s's tokens.
struct TrampolineLayout {
    long long rows, meta, routes, total;
};
TrampolineLayout trampoline_layout(const Dims& d);
cudaError_t launch_dispatch_trampoline(const Dims& d, const uint16_t* x, const int32_t* phys_idx,
                                       void* tbuf, void* dbuf, long long meta_off,
                                       int32_t* rank_counts, int32_t* expert_offsets,
                                       int32_t* expert_rows, void* ws, const WsLayout& wl,
                                       cudaStream_t st);

// MOE_OK for cudaSuccess, else MOE_ERR_CUDA with the error kept for
// moe_last_cuda_error.
moe_status record_cuda_status(cudaError_t e);

// Optional kernel timing: when enabled, the expert GEMM launches are
// bracketed by CUDA events (slot 0: gate/up GEMM, slot 1: down GEMM; slots 2
// and 3: the matrix-vector kernels of the narrow experts beside the
// tensor-core GEMMs), and so are the four steps inside moe_layer (slots 4..7:
// route, dispatch, expert FFN, combine).
constexpr int kProfSlots = 8;
cudaEvent_t prof_event(int slot, int end);  // nullptr when profiling is off

// Kernel launchers (each returns cudaGetLastError() after its launches).
cudaError_t launch_route(const Dims& d, const float* logits, const int32_t* rep_table,
                         const int32_t* n_copies, int max_copies, int32_t* topk_idx,
                         float* topk_w, int32_t* phys_idx, int32_t* expert_counts,
                         cudaStream_t st);
// FusedDispatch; with `clear` the workspace status word is cleared first.
// With `stage_rows` (moe_layer, tensor-core FFN next, INT8 messages) the
// scatter also writes the tensor-core FFN's input rows into the workspace:
// the fp16 codes of each message at its expert-row position and its scale,
// what the FFN's assembly step would compute from the messages.
cudaError_t launch_dispatch(const Dims& d, const uint16_t* x, const int32_t* phys_idx,
                            void* dbuf, long long meta_off, int32_t* rank_counts,
                            int32_t* expert_offsets, int32_t* expert_rows, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear = true,
                            bool stage_rows = false);
cudaError_t launch_combine(const Dims& d, const void* cbuf, long long scale_off,
                           const float* topk_w, uint16_t* out, cudaStream_t st);
// CUDA-core grouped GEMM; row_index entries must lie in [0, a_rows), weight
// sets in [0, n_sets) (else MOE_ERR_INDEX is posted to *err).
cudaError_t launch_grouped_gemm_s8(int n_groups, const int32_t* offsets, long long max_rows,
                                   const int32_t* row_index, long long a_rows, const int8_t* A,
                                   long long lda, const int8_t* B, long long b_group_stride,
                                   const int32_t* group_to_set, int n_sets, int N, int K, int32_t* C,
                                   int32_t* tile_prefix, int* err, cudaStream_t st);
// Exclusive prefix of the token tiles (at most BM rows) of each of G groups,
// tile_prefix[G] = their total; with a non-null `table`, also one entry per
// token tile: (weight set = g2s[g] or g, first row, rows, group g).  Offsets
// that are not a nondecreasing prefix from 0 to at most max_rows, or a weight
// set outside [0, n_sets), give no tiles and post MOE_ERR_INDEX to *err.
// Groups with 1..skip_rows rows get no tile (another kernel takes them); with
// a non-null `narrow`, their ids go to narrow[1..] and their number to
// narrow[0].
cudaError_t launch_tile_prefix(int G, int BM, const int32_t* offsets, long long max_rows, int n_sets,
                               int32_t* tile_prefix, int* err, cudaStream_t st,
                               int4* table = nullptr, const int32_t* g2s = nullptr, int skip_rows = 0,
                               int32_t* narrow = nullptr);
cudaError_t launch_grouped_gemm_tc(int n_groups, const int32_t* offsets, long long max_rows,
                                   const int32_t* row_index, const int8_t* A, long long lda,
                                   const int8_t* B, int N, int K, int32_t* C, void* ws,
                                   cudaStream_t st);
// The expert FFN launchers clear the workspace status word first when
// `clear` is set (moe_layer clears it once, before the dispatch).
cudaError_t launch_ffn_simt(const Dims& d, const void* dbuf, long long meta_off,
                            const int32_t* expert_offsets, const int32_t* expert_rows,
                            const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear);
// FusedCombine folded into the expert FFN (INT8 return messages, tensor-core
// path): gate weights, the output, the contributions each token's combine
// waits for (k) and the bound of that wait.  Null members: no fusion.
struct FusedCombine {
    const float* topk_w;  // [T][k]
    uint16_t* out;        // bf16 [T][H]
    int expected = 0;
    unsigned long long wait_ns = 0;
};
// rows_ready: the input rows and their scales are in the workspace already
// (written by a staging dispatch), so the assembly step is skipped.
cudaError_t launch_ffn_tc(const Dims& d, const void* dbuf, long long meta_off,
                          const int32_t* expert_offsets, const int32_t* expert_rows,
                          const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                          const WsLayout& wl, cudaStream_t st, const FusedCombine& fc, bool clear,
                          bool rows_ready = false);
// fp16 copy of an int8 array (moe_weights_to_f16).
cudaError_t launch_weights_to_f16(const int8_t* src, long long n, uint16_t* dst, cudaStream_t st);
// SwiGLU and the token-wise requantisation of its output (row kernel of the
// tensor-core and matrix-vector paths): h = SiLU(g) * u from g, u [M][2I],
// hq as exact fp16 integers and the scales s_h; it also zeroes each row's
// word of ymax, which the down projection's epilogue then max-reduces.
cudaError_t launch_requant_rows(int I, long long M, const float* gu, void* hq16, float* sh, unsigned* ymax,
                                cudaStream_t st);
// INT8 return messages from y and its row maxima into the combine rows
// (rows whose dispatch slot or metadata is out of range are skipped and
// MOE_ERR_INDEX is posted to *err).
cudaError_t launch_retquant_rows(const Dims& d, long long M, const float* y, const unsigned* rowmax,
                                 const int32_t* expert_rows, const moe_dispatch_meta* meta,
                                 unsigned char* cbuf, float* cscale, int* err, cudaStream_t st);
// Decode batches (at most kGemvRowsPerExpert routed rows per expert on
// average, INT8 return messages, H and I multiples of 512): the expert FFN
// by streamed CUDA-core matrix-vector products, same outputs as launch_ffn_tc.
bool ffn_gemv_fits(const Dims& d);
// Whether the matrix-vector kernels apply to the shape at all (INT8 return
// messages, H and I multiples of 512, token rows within shared memory).
bool gemv_kernels_fit(const Dims& d);
// Rows up to which an expert runs on the matrix-vector kernels beside the
// tensor-core GEMMs (0: none).
inline int narrow_expert_rows(const Dims& d) { return gemv_kernels_fit(d) ? kNarrowExpertRows : 0; }
// The matrix-vector kernels on their own, writing g and u / y and the row
// maxima of y exactly as the tensor-core epilogues do: every expert (list ==
// nullptr), or the experts listed in list[1..list[0]]; prof_slot selects the
// timing events.
cudaError_t launch_gemv_gate_up(const Dims& d, const void* dbuf, const moe_dispatch_meta* meta,
                                const int32_t* expert_offsets, const int32_t* expert_rows,
                                const moe_expert_weights& w, float* gubuf, int* err,
                                const int32_t* list, int prof_slot, cudaStream_t st);
cudaError_t launch_gemv_down(const Dims& d, const int32_t* expert_offsets, const moe_expert_weights& w,
                             const void* hq16, const float* sh, float* ybuf, unsigned* ymax, int* err,
                             const int32_t* list, int prof_slot, cudaStream_t st);
cudaError_t launch_ffn_gemv(const Dims& d, const void* dbuf, long long meta_off,
                            const int32_t* expert_offsets, const int32_t* expert_rows,
                            const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                            const WsLayout& wl, cudaStream_t st, bool clear);
// Whether launch_ffn performs the combine itself for this shape.
inline bool ffn_fuses_combine(const Dims& d, const WsLayout& wl) {
    return wl.tc && d.cfmt == MOE_MSG_INT8;
}
inline cudaError_t launch_ffn(const Dims& d, const void* dbuf, long long meta_off,
                              const int32_t* expert_offsets, const int32_t* expert_rows,
                              const moe_expert_weights& w, void* cbuf, long long scale_off, void* ws,
                              const WsLayout& wl, cudaStream_t st,
                              const FusedCombine& fc = FusedCombine{nullptr, nullptr},
                              bool clear = true, bool rows_ready = false) {
    if (!wl.tc)
        return launch_ffn_simt(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf, scale_off, ws,
                               wl, st, clear);
    if (fc.out == nullptr && ffn_gemv_fits(d))
        return launch_ffn_gemv(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf, scale_off, ws,
                               wl, st, clear);
    return launch_ffn_tc(d, dbuf, meta_off, expert_offsets, expert_rows, w, cbuf, scale_off, ws, wl,
                         st, fc, clear, rows_ready);
}
// Whether launch_ffn takes the tensor-core GEMMs (and reads the staged
// expert input rows) for this shape without a fused combine.
inline bool ffn_takes_tc(const Dims& d, const WsLayout& wl) { return wl.tc && !ffn_gemv_fits(d); }

}  // namespace moe
