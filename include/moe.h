/*
 * moe.h -- C ABI of the GB300 (sm_103a) decode-time MoE layer library.
 *
 * The library computes one DeepSeek-V3/R1-shaped MoE layer on one GPU:
 *   moe_route       gate top-k + renormalised softmax weights + EPLB
 *                   logical->physical map + per-expert counts
 *   moe_dispatch    FusedDispatch: token-wise INT8 quantisation fused with the
 *                   scatter of one message per (token, route) into static
 *                   per-rank buffers, plus the per-expert row lists
 *   moe_expert_ffn  grouped W8A8 SwiGLU expert FFN reading the dispatch
 *                   buffer and writing one return message per (token, route)
 *   moe_combine     FusedCombine: dequantise and gate-weighted sum
 *   moe_layer       the four steps above, in order, on one stream
 * "Ranks" are partitions of this GPU's memory: source rank s owns tokens
 * [s*lb, (s+1)*lb), destination rank d owns physical experts
 * [d*epr, (d+1)*epr).  There are no collectives.
 *
 * Sources (page title, section):
 *   [X] "xDeepServe on CloudMatrix384": "合设 MoE-Attention 的 All-to-All"
 *       (P038-P041, DISPATCH/COMBINE procedures), "专家负载均衡" (P068-P079),
 *       "DeepSeek INT8 量化" (P085 equation, P088, P089).
 *   [C] "CloudMatrix384 LLM Serving": "EP320：token 去找专家" (fused_moe
 *       listing), "缓冲区公式" (max_tokens and buffer_size equations).
 *
 * Conventions for every entry point:
 *   - The caller owns all memory.  Pointers marked (device) are CUDA device
 *     pointers on the current device; (host) are host pointers.  The library
 *     never allocates and never synchronises the stream; work is enqueued on
 *     `stream` (a cudaStream_t; NULL is the legacy default stream) and the
 *     call returns before it runs.
 *   - Arguments are validated on the host before anything is enqueued;
 *     a failure returns MOE_ERR_INVALID_ARG (bad shape, null pointer,
 *     misaligned buffer) or MOE_ERR_WORKSPACE (a buffer smaller than
 *     moe_query_layout reports) and enqueues nothing.
 *   - MOE_ERR_CUDA means a launch failed; the stream may hold part of the
 *     work.
 *   - Device-side checks.  Every index the kernels take from a caller's
 *     device array (physical expert ids, replica-table entries, row lists,
 *     offsets, message metadata, weight-set ids) is checked against its
 *     range before it addresses memory.  A bad index never leads to an
 *     access outside the caller's buffers: the access is skipped (or made
 *     on an in-range element whose result is meaningless) and a code is
 *     posted to the device status word at the start of the workspace,
 *     read with moe_device_status:
 *       MOE_ERR_INDEX     an index outside its range (the outputs of that
 *                         call are unspecified);
 *       MOE_ERR_CAPACITY  a (destination, source) pair received more than
 *                         max_tokens messages, which only a replica table
 *                         that maps two routes of one token onto one
 *                         physical expert can cause (the extra messages are
 *                         dropped);
 *       MOE_ERR_TIMEOUT   a bounded device wait gave up.
 *     The first code posted stays.  Each entry point that takes a
 *     workspace clears the word when its work starts on the stream
 *     (moe_layer once, for the whole layer), so the word describes the most
 *     recent such call.
 *   - Device buffers passed as `void*` must be 256-byte aligned.
 *   - All integer outputs (indices, counts, offsets, slots, INT8 codes, int32
 *     accumulators) are deterministic and bit-exact with respect to the
 *     written definitions below; float outputs follow the stated operation
 *     order.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_WORKSPACE = 2,
    MOE_ERR_CAPACITY = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_TIMEOUT = 5,
    MOE_ERR_UNSUPPORTED = 6,
    MOE_ERR_INDEX = 7
} moe_status;

/* Message formats ([X] P041/P089: INT8 halves message bytes; bf16 is the
 * unquantised form). */
typedef enum { MOE_MSG_BF16 = 0, MOE_MSG_INT8 = 1 } moe_msg_format;

/* Layer shape.  Limits checked by every entry point:
 *   1 <= T, 16 <= H <= 16384 and H % 16 == 0, 16 <= I <= 16384 and
 *   I % 16 == 0, 1 <= k <= min(E_log, 32), E_log <= E_phys <= 1024,
 *   E_phys % n_ranks == 0, T % n_src_ranks == 0, T * k < 2^31. */
typedef struct {
    int32_t T;            /* tokens in the batch */
    int32_t H;            /* hidden size */
    int32_t E_log;        /* logical (routed) experts */
    int32_t E_phys;       /* physical expert slots = E_log + redundant slots */
    int32_t k;            /* experts per token (top-k) */
    int32_t I;            /* SwiGLU intermediate size per expert */
    int32_t n_ranks;      /* R: destination ranks, epr = E_phys / R experts each */
    int32_t n_src_ranks;  /* S: source ranks, lb = T / S tokens each */
    int32_t dispatch_fmt; /* moe_msg_format of dispatch messages */
    int32_t combine_fmt;  /* moe_msg_format of return (combine) messages */
} moe_shape;

/* Metadata that travels with every dispatch message ([C] fused_moe listing:
 * scale, source_rank, batch_slot, route_slot).  16 bytes. */
typedef struct {
    float scale;        /* token scale (INT8 messages), 0 for bf16 messages */
    int32_t src_rank;   /* source rank s */
    int32_t batch_slot; /* token index within the source rank, t - s*lb */
    int32_t route_slot; /* j: position of the expert in the token's top-k */
} moe_dispatch_meta;

/* Sizes and offsets of the caller-owned buffers for one shape.
 *
 * Dispatch buffer ([C] "缓冲区公式"): for each destination rank d, a static
 * area of n_src_ranks * max_tokens messages, max_tokens = lb * min(k, epr):
 *   rows: [R][S][max_tokens][dispatch_row_bytes] at offset 0, where a row is
 *         H INT8 codes or H bf16 values;
 *   meta: [R][S][max_tokens] moe_dispatch_meta at dispatch_meta_offset.
 *   Message (t, j) to rank d from source s sits in slot
 *   g = (d*S + s)*max_tokens + n, n counting that pair's messages in
 *   ascending (batch_slot, route_slot) order.
 * Combine buffer ([C]: results are written back to (source_rank, batch_slot,
 * route_slot)): rows [T][k][combine_row_bytes] at offset 0 (H INT8 codes or
 * H bf16 values), and for INT8 one float scale per row, [T][k] at
 * combine_scale_offset.
 * Workspace: scratch for the library's kernels, workspace_bytes covers every
 * entry point for this shape (moe_layer included). */
typedef struct {
    int64_t max_tokens;           /* lb * min(k, epr) */
    int64_t dispatch_row_bytes;   /* H or 2H */
    int64_t dispatch_meta_offset; /* bytes */
    int64_t dispatch_bytes;       /* total dispatch buffer bytes */
    int64_t combine_row_bytes;    /* H or 2H */
    int64_t combine_scale_offset; /* bytes; equals combine rows bytes */
    int64_t combine_bytes;        /* total combine buffer bytes */
    int64_t workspace_bytes;      /* scratch bytes */
} moe_layout;

/* Which kernels moe_expert_ffn and moe_layer run the expert FFN with for
 * `shape` (host only; moe_expert_ffn_combine always takes the tensor-core
 * GEMMs where the shape allows them).  The choice depends on the shape alone:
 *   MOE_FFN_CUDA_CORE    H or I not a multiple of 64: dp4a grouped GEMMs;
 *   MOE_FFN_TENSOR_CORE  the exact-int8 tcgen05 grouped GEMMs;
 *   MOE_FFN_GEMV         decode batches (INT8 return messages, H and I
 *                        multiples of 512, T*k at most 4 rows per physical
 *                        expert): weight-streaming matrix-vector products.
 * All three give the same outputs bit for bit.  INVALID_ARG for a bad shape
 * or a null `path`. */
enum { MOE_FFN_CUDA_CORE = 0, MOE_FFN_TENSOR_CORE = 1, MOE_FFN_GEMV = 2 };
moe_status moe_expert_ffn_path(const moe_shape* shape, int32_t* path);

/* On the tensor-core path, physical experts with 1 to *rows routed rows are
 * computed by the weight-streaming matrix-vector kernels instead, in the
 * same launch sequence and with the same outputs bit for bit: for an expert
 * with a handful of tokens the tensor-core pipeline spends its time
 * converting the expert's whole weight matrix, while the matrix-vector
 * kernels stream it at the memory roofline.  *rows is 8 where those kernels
 * apply (INT8 return messages, H and I multiples of 512), else 0 (and 0 when
 * the whole FFN already runs on them, MOE_FFN_GEMV).  Host only. */
moe_status moe_expert_ffn_narrow_rows(const moe_shape* shape, int32_t* rows);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* The page's static-buffer formula ([C] "缓冲区公式"):
 *   *bytes = rank_num * (local_batch * min(topk, experts_per_rank)) * msg_size.
 * Host only.  INVALID_ARG if any input is < 1 or the product overflows. */
moe_status moe_static_buffer_bytes(int64_t rank_num, int64_t local_batch, int64_t topk,
                                   int64_t experts_per_rank, int64_t msg_size,
                                   int64_t* bytes);

/* Buffer layout for `shape` (host only). */
moe_status moe_query_layout(const moe_shape* shape, moe_layout* layout);

/* EPLB replica planner ([X] "专家负载均衡", P069-P076), host only.
 * token_count (host) [n_slices][E_log]: tokens routed to each logical expert
 * in each time slice.  Selects E_phys - E_log redundant copies greedily (each
 * round, among the experts that are the hottest of some slice, add a copy to
 * the one whose even split gives the smallest sum over slices of the hottest
 * load; ties to the lower id), then places them heaviest first on the rank
 * with the least load that has a free redundant slot and does not yet host
 * that expert (if none, any rank with a free slot; ties to the lower rank).
 * A rank's load starts as the sum of load/copies of its primary experts.
 * Rank r owns physical slots r*epr .. r*epr+epr-1; the first E_log/R hold
 * logical experts r*(E_log/R)+m, the rest are the redundant slots.
 * Outputs (host): rep_table [E_log][max_copies] (physical ids of each
 * logical expert in ascending order, padded with -1), n_copies [E_log],
 * phys_to_logical [E_phys].  INVALID_ARG if E_log or E_phys is not a
 * multiple of n_ranks, E_phys < E_log, or max_copies is too small. */
moe_status moe_eplb_plan(int32_t n_slices, int32_t E_log, int32_t E_phys, int32_t n_ranks,
                         const double* token_count, int32_t max_copies,
                         int32_t* rep_table, int32_t* n_copies, int32_t* phys_to_logical);

/* Load aggregation of the EPLB loop ([X] "专家负载均衡" P068: the Collect
 * kernel's counts, summed over a time window for the planner).
 *   load[e] += sum of expert_counts[p] over the physical experts p with
 *   phys_to_logical[p] == e, for e in [0, E_log).
 *   expert_counts (device) int32 [E_phys], as moe_route writes it;
 *   phys_to_logical (device) int32 [E_phys], or NULL when E_phys == E_log
 *   (identity); load (device) int64 [E_log], accumulated, never cleared here.
 * Integer sums, so the result does not depend on the order of additions.
 * One small kernel on `stream`; no workspace. */
moe_status moe_eplb_collect(int32_t E_log, int32_t E_phys, const int32_t* expert_counts,
                            const int32_t* phys_to_logical, int64_t* load, moe_stream_t stream);

/* Gate top-k ([X] P038) with renormalised softmax weights and the EPLB map
 * ([X] P078-P079), plus per-physical-expert counts (the Collect kernel of
 * [X] P068).
 *   logits (device) f32 [T][E_log], finite.  A NaN logit is read as -inf, so
 *   that the indices stay valid (the weights of such a row are unspecified).
 *   Selection: logit descending, ties to the lower expert id; topk_idx[t][j]
 *   (device, int32 [T][k]) is the j-th selected logical expert (route_slot j).
 *   topk_w[t][j] (device, f32 [T][k]) = e^(l_j - l_0) / sum_i e^(l_i - l_0)
 *   in binary32.
 *   rep_table (device, nullable) int32 [E_log][max_copies], n_copies (device)
 *   int32 [E_log]: phys_idx[t][j] = rep_table[e][t mod n_copies[e]] for
 *   e = topk_idx[t][j]; with rep_table NULL, phys_idx = topk_idx and
 *   E_phys must equal E_log.  The table must list, for each logical expert
 *   e, n_copies[e] in [1, max_copies] distinct physical slots that hold e;
 *   an entry outside [0, E_phys) or a copy count outside [1, max_copies]
 *   gives phys_idx = -1 for that route (not counted), which moe_dispatch
 *   then reports as MOE_ERR_INDEX.
 *   expert_counts (device) int32 [E_phys]: messages per physical expert,
 *   counted without atomics (per-warp histograms summed across one thread
 *   block cluster).
 * No workspace is used. */
moe_status moe_route(const moe_shape* shape, const float* logits, const int32_t* rep_table,
                     const int32_t* n_copies, int32_t max_copies, int32_t* topk_idx,
                     float* topk_w, int32_t* phys_idx, int32_t* expert_counts,
                     moe_stream_t stream);

/* FusedDispatch ([C] fused_moe listing; [X] DISPATCH procedure, P039-P040).
 *   x (device) bf16 [T][H] (raw 16-bit patterns); phys_idx (device) int32
 *   [T][k] from moe_route.
 *   INT8 messages: per token, scale = absmax/127 (binary32 division), code =
 *   round-half-even(x / scale) clamped to [-127, 127]; a zero row has scale
 *   0 and codes 0.  BF16 messages carry the row unchanged.
 *   Writes each message (t, j) to its slot of dispatch_buf (layout above)
 *   with its moe_dispatch_meta.
 *   rank_counts (device) int32 [R][S]: messages from source s to rank d.
 *   expert_offsets (device) int32 [E_phys+1]: exclusive prefix of messages
 *   per physical expert; expert_rows (device) int32 [T*k]: for each expert,
 *   the slot ids g of its messages in ascending token order (the expert's
 *   gathered input rows, [C] assemble_expert_inputs).
 *   Slots not written keep their previous contents.  Uses the workspace.
 *   A phys_idx entry outside [0, E_phys) drops that message (MOE_ERR_INDEX
 *   in the status word). */
moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* phys_idx,
                        void* dispatch_buf, int64_t dispatch_bytes, int32_t* rank_counts,
                        int32_t* expert_offsets, int32_t* expert_rows, void* workspace,
                        int64_t workspace_bytes, moe_stream_t stream);

/* Expert weights: W8A8 with one binary32 scale per output channel ([X] P085).
 *   w_gate_up (device) int8 [E_w][2I][H]: rows 0..I-1 are gate_proj, I..2I-1
 *   up_proj (fused, [X] P088); s_gate_up (device) f32 [E_w][2I];
 *   w_down (device) int8 [E_w][H][I]; s_down (device) f32 [E_w][H].
 *   phys_to_weight (device, nullable) int32 [E_phys]: weight set of each
 *   physical expert (replicas alias their logical expert); NULL means
 *   physical expert p uses set p (E_w >= E_phys).
 *   w_gate_up_f16, w_down_f16 (device, nullable, both or neither; 16-byte
 *   aligned): fp16 copies of w_gate_up and w_down in the same layout, made
 *   once by moe_weights_to_f16 (every int8 value is exact in fp16).  With
 *   them, batches above the decode size (more than 32 routed rows per
 *   physical expert on average) run the tensor-core GEMMs on the copies
 *   instead of converting int8 weight tiles on the SM: the same results bit
 *   for bit, at twice the weight bytes held and read.  The int8 arrays stay
 *   required (decode batches and experts with few rows read them). */
typedef struct {
    const int8_t* w_gate_up;
    const float* s_gate_up;
    const int8_t* w_down;
    const float* s_down;
    int32_t n_sets; /* E_w */
    const int32_t* phys_to_weight;
    const uint16_t* w_gate_up_f16;
    const uint16_t* w_down_f16;
} moe_expert_weights;

/* dst[i] = the fp16 encoding of the int8 value src[i], i in [0, n): the
 * weight copies of moe_expert_weights.  src and dst (device) 16-byte
 * aligned, n >= 0 (any value; a multiple of 16 takes only vector stores).
 * Enqueued on `stream`; n = 0 does nothing.  INVALID_ARG for n < 0, or for
 * null or misaligned pointers with n > 0. */
moe_status moe_weights_to_f16(const int8_t* src, int64_t n, uint16_t* dst, moe_stream_t stream);

/* Grouped W8A8 SwiGLU expert FFN ([X] P085 equation, P088, P089; [C]
 * run_local_experts and remote_write_combine).  Requires INT8 dispatch
 * messages.  For every routed row (dispatch slot g of physical expert p,
 * codes q, scale s):
 *   acc_g[i] = sum_h q[h] Wg[i][h], acc_u[i] = sum_h q[h] Wu[i][h]  (exact int32)
 *   g = (acc_g * s) * sg[i], u = (acc_u * s) * su[i]   (binary32, two roundings)
 *   h = g / (1 + e(-g)) * u, e the binary32 exp specification: n =
 *       rint(x * RN(1/ln2)), r = (x - n*LN2_HI) - n*LN2_LO with ln 2 split
 *       into a 14-bit head and a tail, e^r by the degree-7 Taylor polynomial
 *       in Horner form, times 2^n; one rounding per operation, no fused
 *       multiply-add; +inf above x = 88, 0 below x = -87
 *   hq, s_h = token-wise INT8 quantisation of h (as in moe_dispatch)
 *   acc_d[c] = sum_i hq[i] Wd[c][i] (exact int32), y = (acc_d * s_h) * sd[c]
 *   return message at combine row (t, j), t = src_rank*lb + batch_slot,
 *   j = route_slot: INT8 codes of y + scale (combine_fmt INT8) or bf16(y).
 * Uses the workspace. */
moe_status moe_expert_ffn(const moe_shape* shape, const void* dispatch_buf,
                          int64_t dispatch_bytes, const int32_t* expert_offsets,
                          const int32_t* expert_rows, const moe_expert_weights* weights,
                          void* combine_buf, int64_t combine_bytes, void* workspace,
                          int64_t workspace_bytes, moe_stream_t stream);

/* FusedCombine ([C] fused_moe listing; [X] COMBINE procedure):
 *   out[t][h] = bf16_rne( sum_{j=0..k-1} topk_w[t][j] * v[t][j][h] )
 * with v = code * scale (INT8) or the bf16 value, the sum taken in binary32
 * in ascending j: for INT8 each term adds RN(topk_w * scale) * code by one
 * fused multiply-add; for bf16 the product and the sum are rounded
 * separately.
 *   topk_w (device) f32 [T][k]; out (device) bf16 [T][H].  No workspace. */
moe_status moe_combine(const moe_shape* shape, const void* combine_buf, int64_t combine_bytes,
                       const float* topk_w, uint16_t* out, moe_stream_t stream);

/* moe_expert_ffn and moe_combine in one pass, with the combine of each token
 * started once its k return messages are in ([C] "EP320" fused_moe listing:
 * combine waits until all contributions have arrived; [X] COMBINE
 * procedure).  After the two expert GEMMs, one persistent kernel (cooperative
 * launch, every block resident) takes work items from an atomic ticket in
 * the workspace: first the T*k expert rows, then the T tokens.  A row's
 * block writes its INT8 return message, fences and increments the token's
 * readiness counter; a token's block waits, with a bounded spin on
 * %globaltimer, until the counter reaches k, then sums the k messages and
 * writes out[t].  Every row is taken before any token by a block that waits
 * for nothing, so each wait ends once the rows are written.  Same outputs as
 * moe_expert_ffn followed by moe_combine, bit for bit (combine_buf holds the
 * messages too).
 *   Arguments: those of moe_expert_ffn plus topk_w and out of moe_combine.
 *   UNSUPPORTED unless combine_fmt is MOE_MSG_INT8 and the tensor-core path
 *   applies (H and I multiples of 64).
 * A wait that reaches its bound (2 s; only a lost message can cause it)
 * posts MOE_ERR_TIMEOUT to the status word and skips that token; once any
 * error is posted the remaining waits give up at once, so the kernel always
 * ends.  moe_layer keeps the separate calls (faster on the measured
 * workloads: the last return messages of a token come late in the launch). */
moe_status moe_expert_ffn_combine(const moe_shape* shape, const void* dispatch_buf,
                                  int64_t dispatch_bytes, const int32_t* expert_offsets,
                                  const int32_t* expert_rows, const moe_expert_weights* weights,
                                  const float* topk_w, void* combine_buf, int64_t combine_bytes,
                                  uint16_t* out, void* workspace, int64_t workspace_bytes,
                                  moe_stream_t stream);
/* moe_expert_ffn_combine with the wait's target and bound given: each token's
 * combine waits until `expected` (>= 1; k for the layer) messages are in, at
 * most wait_ns (>= 1) nanoseconds.  A target no token can reach (more than k)
 * makes the first wait run out, post MOE_ERR_TIMEOUT and return; this is the
 * path a lost message would take, and the call still completes. */
moe_status moe_expert_ffn_combine_ex(const moe_shape* shape, const void* dispatch_buf,
                                     int64_t dispatch_bytes, const int32_t* expert_offsets,
                                     const int32_t* expert_rows, const moe_expert_weights* weights,
                                     const float* topk_w, void* combine_buf, int64_t combine_bytes,
                                     uint16_t* out, void* workspace, int64_t workspace_bytes,
                                     int32_t expected, int64_t wait_ns, moe_stream_t stream);

/* Routing arrays produced inside moe_layer (all device, caller-owned). */
typedef struct {
    int32_t* topk_idx;       /* [T][k] */
    float* topk_w;           /* [T][k] */
    int32_t* phys_idx;       /* [T][k] */
    int32_t* expert_counts;  /* [E_phys] */
    int32_t* rank_counts;    /* [R][S] */
    int32_t* expert_offsets; /* [E_phys+1] */
    int32_t* expert_rows;    /* [T*k] */
} moe_routing;

/* The whole layer: moe_route -> moe_dispatch -> moe_expert_ffn ->
 * moe_combine on one stream, with the same definitions and outputs.  When the
 * expert FFN takes the tensor-core GEMMs (moe_expert_ffn_path), the dispatch
 * kernel also writes the FFN's input rows (the fp16 codes of each message at
 * its position in the expert row lists, with its scale) into the workspace,
 * and the FFN skips the assembly step that would read them back from the
 * dispatch buffer ([C] assemble_expert_inputs, fused into the dispatch).
 * Under MOE_ERR_CAPACITY the row of a dropped message then holds that
 * token's codes rather than a copy of another message (the outputs of such a
 * call are unspecified either way).  rep_table / n_copies may be NULL (no
 * replicas). */
moe_status moe_layer(const moe_shape* shape, const float* logits, const uint16_t* x,
                     const int32_t* rep_table, const int32_t* n_copies, int32_t max_copies,
                     const moe_expert_weights* weights, const moe_routing* routing,
                     void* dispatch_buf, int64_t dispatch_bytes, void* combine_buf,
                     int64_t combine_bytes, void* workspace, int64_t workspace_bytes,
                     uint16_t* out, moe_stream_t stream);

/* The whole layer from host memory to host memory: on `stream`, copies
 * h_logits (host, f32 [T][E_log]) into d_logits (device, same shape) and h_x
 * (host, bf16 [T][H]) into d_x (device), runs moe_layer on them with the
 * other arguments as moe_layer takes them, and copies the output d_out
 * (device, bf16 [T][H]) back into h_out (host).  One cudaMemcpyAsync per
 * copy; nothing is allocated and the stream is not synchronised: h_out holds
 * the result once `stream` has reached that point.  Host buffers should be
 * page-locked (cudaHostAlloc or cudaHostRegister), or the copies may block
 * the calling thread.  A serving loop overlaps one step's copies with
 * another step's kernels by alternating two streams and two sets of device
 * buffers (the host input may be shared; each set needs its own h_out).
 * Argument errors are those of moe_layer plus null or misaligned (16-byte)
 * d_logits / d_x / host pointers. */
moe_status moe_layer_host(const moe_shape* shape, const float* h_logits, const uint16_t* h_x,
                          uint16_t* h_out, float* d_logits, uint16_t* d_x, const int32_t* rep_table,
                          const int32_t* n_copies, int32_t max_copies,
                          const moe_expert_weights* weights, const moe_routing* routing,
                          void* dispatch_buf, int64_t dispatch_bytes, void* combine_buf,
                          int64_t combine_bytes, void* workspace, int64_t workspace_bytes,
                          uint16_t* d_out, moe_stream_t stream);

/* The decode layer as a CUDA graph ([C] "EP320：token 去找专家": the static
 * dispatch/combine buffers are allocated once, reused by every decode step
 * and double-buffered so that one step's combine cannot overwrite dispatch
 * data another step still uses).
 *   moe_layer_graph_create captures one moe_layer call with exactly these
 *   arguments on `capture_stream` and instantiates it; nothing runs during
 *   the call.  Each moe_graph_launch then replays the whole layer on
 *   `stream` with the same buffers, reading whatever `logits` and `x` hold
 *   when it runs and writing the same outputs moe_layer writes.  Double
 *   buffering is two graphs over two buffer sets, launched in turn.
 *   - capture_stream (a cudaStream_t) must not be NULL (the legacy default
 *     stream cannot be captured) and must not be capturing already; the
 *     capture uses cudaStreamCaptureModeThreadLocal.
 *   - Argument errors are those of moe_layer and are reported before
 *     anything is captured; *graph is NULL on any error.
 *   - The handle owns the driver's executable graph (host-side objects; no
 *     device buffer is allocated) until moe_graph_destroy.  Buffers passed
 *     here must stay valid while the graph exists.
 *   - Replays of one graph on several streams at once race on its buffers.
 *   - Profiling (moe_profile_enable) should be off while capturing. */
typedef struct moe_graph_s* moe_graph;
moe_status moe_layer_graph_create(const moe_shape* shape, const float* logits, const uint16_t* x,
                                  const int32_t* rep_table, const int32_t* n_copies,
                                  int32_t max_copies, const moe_expert_weights* weights,
                                  const moe_routing* routing, void* dispatch_buf,
                                  int64_t dispatch_bytes, void* combine_buf, int64_t combine_bytes,
                                  void* workspace, int64_t workspace_bytes, uint16_t* out,
                                  moe_stream_t capture_stream, moe_graph* graph);
moe_status moe_graph_launch(moe_graph graph, moe_stream_t stream);
/* NULL is accepted and ignored. */
moe_status moe_graph_destroy(moe_graph graph);

/* Exact grouped INT8 GEMM with int32 output -- the contraction inside
 * moe_expert_ffn ([X] P085: sum_k q(x_ik) q(w_jk)), exposed on its own.
 * With K % 64 == 0 it runs the same tensor-core kernel as moe_expert_ffn
 * (fp16 operands, fp32 accumulation drained to int32 every 1024 K, which is
 * exact); otherwise a CUDA-core dp4a kernel.
 *   For group gi in [0, n_groups) and rows r in [offsets[gi], offsets[gi+1]):
 *     C[r][n] = sum_{kk<K} A[arow(r)][kk] * B[gi][n][kk]     (exact int32)
 *   arow(r) = row_index[r] if row_index != NULL, else r.
 *   offsets (device) int32 [n_groups+1], nondecreasing, offsets[0] = 0,
 *   offsets[n_groups] = M_total <= max_rows; A (device) int8 rows of lda
 *   bytes; B (device) int8 [n_groups][N][K]; C (device) int32 [M_total][N].
 *   K % 16 == 0, N % 16 == 0, lda % 16 == 0, lda >= K, K < 2^20.
 *   max_rows bounds M_total (it sizes the launch).  Uses the workspace
 *   (at least moe_gemm_workspace_bytes(n_groups, max_rows, K)). */
int64_t moe_gemm_workspace_bytes(int32_t n_groups, int64_t max_rows, int32_t K);
moe_status moe_grouped_gemm_s8(int32_t n_groups, const int32_t* offsets, int64_t max_rows,
                               const int32_t* row_index, const int8_t* A, int64_t lda,
                               const int8_t* B, int32_t N, int32_t K, int32_t* C,
                               void* workspace, int64_t workspace_bytes, moe_stream_t stream);

/* FusedDispatch by trampoline forward ([X] "合设 MoE-Attention 的
 * All-to-All" P044-P045, P109: with fewer attention ranks than expert ranks,
 * as many expert ranks as there are attention ranks first receive all of an
 * attention rank's data and forward it to the other expert ranks).  Source
 * rank s (an attention rank) uses expert rank s as its trampoline:
 *   hop 1 (A2E):  every token of s is written once into trampoline s's area:
 *                 its message row (INT8 codes + scale, or bf16), its
 *                 batch_slot and its k physical expert ids;
 *   hop 2 (A2E'): the trampoline writes one message per (token, route) into
 *                 the owner's static area.
 * The outputs (dispatch buffer rows and meta, rank_counts, expert_offsets,
 * expert_rows) are those of moe_dispatch, bit for bit.  Requires
 * n_src_ranks <= n_ranks.
 *   trampoline_buf (device, 256-byte aligned) of moe_trampoline_bytes bytes:
 *   rows [T][row bytes], then meta [T] (moe_dispatch_meta, route_slot = k),
 *   then routes [T][k] int32, each region 256-byte aligned.  Caller-owned;
 *   its contents after the call are the trampolines' receive areas. */
moe_status moe_trampoline_bytes(const moe_shape* shape, int64_t* bytes);
moe_status moe_dispatch_trampoline(const moe_shape* shape, const uint16_t* x, const int32_t* phys_idx,
                                   void* trampoline_buf, int64_t trampoline_bytes,
                                   void* dispatch_buf, int64_t dispatch_bytes, int32_t* rank_counts,
                                   int32_t* expert_offsets, int32_t* expert_rows, void* workspace,
                                   int64_t workspace_bytes, moe_stream_t stream);

/* FusedDispatch without a workspace.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot call cudaMalloc at all --
 * an engine whose allocator has reserved all device memory and forbids any
 * allocation outside its pool, a latency-critical decode loop that must not
 * risk the synchronisation an allocation or free can bring, a plug-in inside
 * a host process that owns every device-memory decision.
 * Same arguments, definitions and outputs as moe_dispatch, minus the
 * workspace: its scratch (slot/rank arrays and per-source histograms) lives
 * in a file-scope device array of moe_dispatch_noalloc_max_scratch() bytes
 * (4 MiB) that every GPU loading this library holds until the process exits.
 * Allocates nothing and calls no allocating routine.
 *   - A shape whose dispatch scratch exceeds that size (about
 *     8*T*k + 8*n_src_ranks*E_phys + 256 bytes) returns MOE_ERR_WORKSPACE
 *     before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs clearing: every word is written before it is
 *     read).  Calls that overlap on the GPU -- several streams, or several
 *     host threads -- race on it; serialise them. */
moe_status moe_dispatch_noalloc(const moe_shape* shape, const uint16_t* x, const int32_t* phys_idx,
                                void* dispatch_buf, int64_t dispatch_bytes, int32_t* rank_counts,
                                int32_t* expert_offsets, int32_t* expert_rows, moe_stream_t stream);
int64_t moe_dispatch_noalloc_max_scratch(void);

/* Reads the device status word that the library's kernels keep at the start
 * of `workspace` (device): MOE_OK, or the first code a device-side check
 * posted (MOE_ERR_INDEX, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT; see the
 * conventions at the top) during the most recent call that used this
 * workspace.  Synchronises `stream`. */
moe_status moe_device_status(const void* workspace, int32_t* status, moe_stream_t stream);

/* Text of the CUDA error behind the last MOE_ERR_CUDA returned on the
 * calling host thread ("no error" if there was none).  Host only. */
const char* moe_last_cuda_error(void);

/* Optional kernel timing for benchmarks (host only).  While enabled, each
 * tensor-core expert GEMM launch (or matrix-vector kernel of the decode
 * path, see moe_expert_ffn_path) is bracketed by CUDA events on its stream;
 * moe_profile_read synchronises on them and returns the durations (ms) of
 * the most recent gate/up kernel (ms[0]) and down kernel (ms[1]), of the
 * matrix-vector kernels that took the narrow experts beside the tensor-core
 * GEMMs (ms[2] gate/up, ms[3] down; see moe_expert_ffn_narrow_rows), and of
 * the four steps of the most recent moe_layer call (ms[4] route, ms[5]
 * dispatch, ms[6] expert FFN, ms[7] combine: inside moe_layer the dispatch
 * also writes the tensor-core FFN's fp16 input rows, which the FFN then does
 * not assemble); -1 for anything not run since profiling was enabled.
 * n (>= 1) values are written, at most 8 of them meaningful. */
moe_status moe_profile_enable(int32_t on);
moe_status moe_profile_read(float* ms, int32_t n);

/* Number of GPU operations (kernel launches and memsets) the library has
 * enqueued in this process since it was loaded.  Host only, thread-safe. */
int64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
