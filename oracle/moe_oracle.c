/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU reference for the
 * decode-time MoE layer (route -> FusedDispatch -> W8A8 SwiGLU experts ->
 * FusedCombine).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; it is used by the tests, by the smoke check and by the
 * CPU-baseline leg of the benchmark.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (page title, section, paragraph/equation/listing):
 *   [X]  "xDeepServe on CloudMatrix384"
 *        - section "合设 MoE-Attention 的 All-to-All" (P038-P041, the
 *          DISPATCH and COMBINE procedures): top-k routing, pack-by-rank,
 *          token-wise INT8 quantisation, counts, weighted combine.
 *        - section "专家负载均衡" (P078-P079, physical(i,e) = R_e[i mod |R_e|]).
 *        - section "DeepSeek INT8 量化" (P085 equation y_ij ~ s_i s^w_j
 *          sum_k q(x_ik) q(w_jk); P088 fused up/gate projection; P089 expert
 *          inputs AND outputs quantised for communication).
 *   [C]  "CloudMatrix384 LLM Serving"
 *        - section "EP320：token 去找专家" (the fused_moe listing: quantise
 *          once per token, one message per (batch_slot, route_slot) carrying
 *          q_token, scale, source_rank, batch_slot, route_slot; combine waits
 *          for all contributions, dequantises and sums with gate weights).
 *        - section "缓冲区公式" (max_tokens = local_batch * min(topK,
 *          experts_per_die); buffer = rank_num * max_tokens * msg_size).
 *
 * Precision choices (the pages fix INT8 codes and nothing else):
 *   - every float step that decides an integer (a quantised code, a top-k
 *     order) is taken in IEEE binary32 with round-to-nearest-even, one
 *     rounding per operation, no contraction (build with -ffp-contract=off);
 *   - routing weights and the final combine sum are computed in binary64;
 *   - exp inside SiLU follows the written exp specification below (binary32
 *     Cody-Waite reduction + degree-7 Taylor polynomial), because SiLU feeds
 *     the INT8 requantisation of the intermediate activation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD 1

/* ---------------------------------------------------------------- bf16 */

static float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (finite inputs). */
static uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* binary64 -> bfloat16, one rounding (nearest, ties to even), finite inputs.
 * Done by splitting the value into the bf16 grid point below and the
 * remainder, all in binary64 (exact for bf16-representable magnitudes). */
static uint16_t orc_f64_to_bf16(double v)
{
    if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    int e;
    frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    double ulp = ldexp(1.0, e - 8);     /* bf16 keeps 8 significant bits */
    double lo = floor(a / ulp) * ulp;   /* exact: a/ulp < 2^8 * 2 */
    double rem = a - lo;
    double r = lo;
    if (rem > 0.5 * ulp) r = lo + ulp;
    else if (rem == 0.5 * ulp) {
        double k = lo / ulp;            /* integer grid index */
        if (fmod(k, 2.0) != 0.0) r = lo + ulp;
    }
    float rf = (float)r;                /* exact: r is on the bf16 grid */
    if (v < 0) rf = -rf;
    uint32_t u;
    memcpy(&u, &rf, 4);
    return (uint16_t)(u >> 16);
}

uint16_t orc_round_f64_to_bf16(double v) { return orc_f64_to_bf16(v); }
uint16_t orc_round_f32_to_bf16(float v) { return orc_f32_to_bf16(v); }

/* ------------------------------------------------------------ exp spec
 * e(x) in binary32, every operation rounded once:
 *   x > 88      -> +inf;    x < -87 -> 0
 *   n = rint(x * RCP_LN2)            (RCP_LN2 = binary32 nearest 1/ln 2)
 *   r = (x - n*LN2_HI) - n*LN2_LO    (LN2_HI has 14 significant bits, so
 *                                      n*LN2_HI is exact for |n| <= 127)
 *   p = 1 + r(1 + r(1/2 + r(1/6 + r(1/24 + r(1/120 + r(1/720 + r/5040))))))
 *       evaluated by Horner from the innermost term, each step a fused
 *       multiply-add p = fma(r, p, c) (one rounding), the coefficients being
 *       the binary32 values nearest 1/m!
 *   e = p * 2^n                       (exact power-of-two scaling)
 * This is Cody and Waite's argument reduction followed by the Taylor series
 * of e^r on |r| <= ln2/2; its error against exp is about one ulp.
 */
float orc_exp_spec(float x)
{
    const float RCP_LN2 = 1.44269502162933349609375f;
    const float LN2_HI = 0.693145751953125f;
    const float LN2_LO = 1.428606765330187e-06f;
    const float c[8] = {1.0f, 1.0f, 0.5f, 1.0f / 6.0f, 1.0f / 24.0f,
                        1.0f / 120.0f, 1.0f / 720.0f, 1.0f / 5040.0f};
    if (x > 88.0f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    float t = x * RCP_LN2;
    float n = rintf(t);
    float a = n * LN2_HI;
    float b = n * LN2_LO;
    float r = x - a;
    r = r - b;
    float p = c[7];
    for (int m = 6; m >= 0; --m)
        p = fmaf(r, p, c[m]);
    int ni = (int)n;
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float s;
    memcpy(&s, &bits, 4);
    return p * s;
}

/* SiLU(g) = g / (1 + e(-g))  (the SwiGLU gate of DeepSeek's expert FFN). */
float orc_silu(float g)
{
    float d = 1.0f + orc_exp_spec(-g);
    return g / d;
}

/* ------------------------------------------------------- quantisation
 * Token-wise symmetric INT8 ([X] P085, [C] FusedDispatch): one scale per
 * row, scale = absmax / 127, code = round-half-even(v / scale), clamped to
 * [-127, 127]; an all-zero row gets scale 0 and codes 0. */
void orc_quantize_row_f32(int n, const float* v, int8_t* q, float* scale)
{
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(v[i]);
        if (m > a) a = m;
    }
    if (a == 0.0f) {
        for (int i = 0; i < n; ++i) q[i] = 0;
        *scale = 0.0f;
        return;
    }
    float s = a / 127.0f;
    for (int i = 0; i < n; ++i) {
        float z = v[i] / s;
        float r = rintf(z);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    *scale = s;
}

void orc_quantize_rows_bf16(int rows, int H, const uint16_t* x, int8_t* q,
                            float* scale)
{
    float* tmp = (float*)malloc(sizeof(float) * (size_t)H);
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h) tmp[h] = orc_bf16_to_f32(x[(size_t)r * H + h]);
        orc_quantize_row_f32(H, tmp, q + (size_t)r * H, scale + r);
    }
    free(tmp);
}

/* ------------------------------------------------------------- routing
 * Gate top-k ([X] P038: each token goes to its top-k experts by gating
 * score).  Selection key: logit descending, expert id ascending on ties;
 * route_slot j is the j-th selected expert.  Weights: softmax over the k
 * selected logits (renormalised), in binary64, rounded to binary32.
 * Optional EPLB map ([X] P078-P079): phys = R_e[t mod |R_e|], R_e listed in
 * ascending physical id in rep_table[e * max_copies + c].
 * expert_counts[p] = number of (t, j) routed to physical expert p (the
 * Collect kernel of [X] P068). */
int orc_route(int T, int E_log, int E_phys, int k, const float* logits,
              const int32_t* rep_table, const int32_t* n_copies, int max_copies,
              int32_t* topk_idx, float* topk_w, int32_t* phys_idx,
              int32_t* expert_counts)
{
    if (k < 1 || k > E_log) return ORC_BAD;
    unsigned char* taken = (unsigned char*)malloc((size_t)E_log);
    double* z = (double*)malloc(sizeof(double) * (size_t)k);
    for (int p = 0; p < E_phys; ++p) expert_counts[p] = 0;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E_log;
        memset(taken, 0, (size_t)E_log);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E_log; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* ties keep lower id */
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
        }
        double l0 = (double)l[topk_idx[(size_t)t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            z[j] = exp((double)l[topk_idx[(size_t)t * k + j]] - l0);
            sum += z[j];
        }
        for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = (float)(z[j] / sum);
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[(size_t)t * k + j];
            int p = e;
            if (rep_table) {
                int nc = n_copies[e];
                p = rep_table[(size_t)e * max_copies + (t % nc)];
            }
            phys_idx[(size_t)t * k + j] = p;
            expert_counts[p] += 1;
        }
    }
    free(taken);
    free(z);
    return ORC_OK;
}

/* ------------------------------------------------------- buffer formula
 * [C] "缓冲区公式": max_tokens = local_batch * min(topK, experts_per_die),
 * buffer_size = rank_num * max_tokens * msg_size. */
int64_t orc_static_buffer_bytes(int64_t rank_num, int64_t local_batch, int64_t topk,
                                int64_t experts_per_rank, int64_t msg_size)
{
    int64_t m = topk < experts_per_rank ? topk : experts_per_rank;
    return rank_num * (local_batch * m) * msg_size;
}

/* ------------------------------------------------------------ dispatch
 * FusedDispatch ([C] fused_moe listing; [X] DISPATCH procedure).
 * Source rank src = t / lb, batch_slot = t mod lb, destination rank
 * dst = phys / epr.  Messages from one source to one destination take
 * consecutive slots in ascending (batch_slot, route_slot) order.  The
 * static buffer is [dst][src][mt][row], mt = lb * min(k, epr).
 * fmt 1 (INT8): row = H codes, meta scale = token scale.
 * fmt 0 (BF16): row = H bf16 values copied, meta scale = 0.
 * rank_counts[dst][src] = messages; expert_offsets = exclusive prefix of
 * per-physical-expert message counts; expert_rows lists, per expert, the
 * global slot id (dst*S + src)*mt + slot of each message, ascending t.
 * slot_of[t*k + j] = global slot id of message (t, j).  `rows` may be NULL
 * (layout and metadata only). */
int orc_dispatch(int T, int H, int E_phys, int k, int R, int S, int fmt,
                 const uint16_t* x, const int32_t* phys_idx,
                 uint8_t* rows, float* meta_scale, int32_t* meta_src,
                 int32_t* meta_bs, int32_t* meta_rs, int32_t* rank_counts,
                 int32_t* expert_offsets, int32_t* expert_rows, int32_t* slot_of)
{
    if (T % S || E_phys % R) return ORC_BAD;
    int lb = T / S, epr = E_phys / R;
    int mt = lb * (k < epr ? k : epr);
    size_t rowb = (size_t)H * (fmt == 1 ? 1 : 2);
    int8_t* q = (int8_t*)malloc((size_t)H);
    float* tmp = (float*)malloc(sizeof(float) * (size_t)H);
    int32_t* cnt_e = (int32_t*)calloc((size_t)E_phys, sizeof(int32_t));
    int32_t* fill = (int32_t*)calloc((size_t)E_phys, sizeof(int32_t));
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < S; ++s) rank_counts[d * S + s] = 0;
    for (int src = 0; src < S; ++src) {
        for (int bs = 0; bs < lb; ++bs) {
            int t = src * lb + bs;
            const uint16_t* xr = x + (size_t)t * H;
            float sc = 0.0f;
            if (fmt == 1) {
                for (int h = 0; h < H; ++h) tmp[h] = orc_bf16_to_f32(xr[h]);
                orc_quantize_row_f32(H, tmp, q, &sc);
            }
            for (int j = 0; j < k; ++j) {
                int p = phys_idx[(size_t)t * k + j];
                int dst = p / epr;
                int slot = rank_counts[dst * S + src]++;
                if (slot >= mt) { free(q); free(tmp); free(cnt_e); free(fill); return ORC_BAD; }
                size_t g = ((size_t)dst * S + src) * mt + slot;
                if (rows) {
                    if (fmt == 1) memcpy(rows + g * rowb, q, (size_t)H);
                    else memcpy(rows + g * rowb, xr, rowb);
                }
                meta_scale[g] = sc;
                meta_src[g] = src;
                meta_bs[g] = bs;
                meta_rs[g] = j;
                slot_of[(size_t)t * k + j] = (int32_t)g;
                cnt_e[p] += 1;
            }
        }
    }
    expert_offsets[0] = 0;
    for (int p = 0; p < E_phys; ++p) expert_offsets[p + 1] = expert_offsets[p] + cnt_e[p];
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int p = phys_idx[(size_t)t * k + j];
            expert_rows[expert_offsets[p] + fill[p]++] = slot_of[(size_t)t * k + j];
        }
    free(q);
    free(tmp);
    free(cnt_e);
    free(fill);
    return ORC_OK;
}

/* --------------------------------------------------------- expert row
 * One routed row through one W8A8 SwiGLU expert ([X] P085 equation, P088
 * fused up/gate, P089 quantised expert output; [C] run_local_experts).
 *   acc_g[i] = sum_h q[h] Wg[i][h],  acc_u[i] = sum_h q[h] Wu[i][h]   (exact)
 *   g = (acc_g * s) * sg[i],  u = (acc_u * s) * su[i]      (binary32)
 *   h_i = SiLU(g) * u; requantise h token-wise -> hq (I codes), s_h
 *   acc_d[c] = sum_i hq[i] Wd[c][i]                                  (exact)
 *   y_c = (acc_d * s_h) * sd[c]                                     (binary32)
 *   message: cfmt 1 -> token-wise INT8 codes of y + scale; cfmt 0 -> bf16(y)
 * w_gu is [2I][H] (rows 0..I-1 gate, I..2I-1 up), w_d is [H][I].
 * Debug outputs may be NULL. */
int orc_expert_row(int H, int I, const int8_t* xq, float xs,
                   const int8_t* w_gu, const float* s_gu,
                   const int8_t* w_d, const float* s_d, int cfmt,
                   void* msg, float* msg_scale,
                   int32_t* acc_gu_dbg, int8_t* hq_dbg, float* sh_dbg,
                   int32_t* acc_d_dbg, float* y_dbg)
{
    float* hv = (float*)malloc(sizeof(float) * (size_t)I);
    int8_t* hq = (int8_t*)malloc((size_t)I);
    float* y = (float*)malloc(sizeof(float) * (size_t)H);
    for (int i = 0; i < I; ++i) {
        int64_t ag = 0, au = 0;
        const int8_t* wg = w_gu + (size_t)i * H;
        const int8_t* wu = w_gu + (size_t)(I + i) * H;
        for (int h = 0; h < H; ++h) {
            ag += (int64_t)xq[h] * wg[h];
            au += (int64_t)xq[h] * wu[h];
        }
        if (acc_gu_dbg) {
            acc_gu_dbg[i] = (int32_t)ag;
            acc_gu_dbg[I + i] = (int32_t)au;
        }
        float g = (float)(int32_t)ag;
        g = g * xs;
        g = g * s_gu[i];
        float u = (float)(int32_t)au;
        u = u * xs;
        u = u * s_gu[I + i];
        float sg = orc_silu(g);
        hv[i] = sg * u;
    }
    float sh;
    orc_quantize_row_f32(I, hv, hq, &sh);
    if (hq_dbg) memcpy(hq_dbg, hq, (size_t)I);
    if (sh_dbg) *sh_dbg = sh;
    for (int c = 0; c < H; ++c) {
        int64_t a = 0;
        const int8_t* wr = w_d + (size_t)c * I;
        for (int i = 0; i < I; ++i) a += (int64_t)hq[i] * wr[i];
        if (acc_d_dbg) acc_d_dbg[c] = (int32_t)a;
        float v = (float)(int32_t)a;
        v = v * sh;
        v = v * s_d[c];
        y[c] = v;
    }
    if (y_dbg) memcpy(y_dbg, y, sizeof(float) * (size_t)H);
    if (cfmt == 1) {
        orc_quantize_row_f32(H, y, (int8_t*)msg, msg_scale);
    } else {
        uint16_t* m = (uint16_t*)msg;
        for (int c = 0; c < H; ++c) m[c] = orc_f32_to_bf16(y[c]);
        if (msg_scale) *msg_scale = 0.0f;
    }
    free(hv);
    free(hq);
    free(y);
    return ORC_OK;
}

/* All routed rows of a batch through their experts, writing the return
 * message of (t, j) at cbuf[t][j] ([C]: remote_write_combine addressed by
 * (source_rank, batch_slot, route_slot)).  xq/xs are the per-token codes and
 * scales; expert weights are given per logical expert through pointer
 * tables; phys_to_logical (nullable) maps replicas to their logical weights. */
int orc_ffn_all(int T, int H, int I, int k, const int8_t* xq, const float* xs,
                const int32_t* phys_idx, const int32_t* phys_to_logical,
                const int8_t* const* w_gu, const float* const* s_gu,
                const int8_t* const* w_d, const float* const* s_d, int cfmt,
                uint8_t* cbuf, float* cscale)
{
    size_t rowb = (size_t)H * (cfmt == 1 ? 1 : 2);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long tj = 0; tj < (long long)T * k; ++tj) {
        int t = (int)(tj / k);
        int p = phys_idx[tj];
        int e = phys_to_logical ? phys_to_logical[p] : p;
        if (!w_gu[e] || !w_d[e]) { bad = 1; continue; }
        orc_expert_row(H, I, xq + (size_t)t * H, xs[t], w_gu[e], s_gu[e], w_d[e],
                       s_d[e], cfmt, cbuf + (size_t)tj * rowb, cscale + tj,
                       NULL, NULL, NULL, NULL, NULL);
    }
    return bad ? ORC_BAD : ORC_OK;
}

/* ------------------------------------------------------------- combine
 * FusedCombine ([C] fused_moe listing; [X] COMBINE procedure):
 * out[t] = sum_j w[t][j] * deq(msg[t][j]), deq = code * scale (INT8) or the
 * bf16 value; summed in binary64, rounded once to bf16. */
int orc_combine(int T, int H, int k, int cfmt, const uint8_t* cbuf,
                const float* cscale, const float* topk_w, uint16_t* out)
{
    size_t rowb = (size_t)H * (cfmt == 1 ? 1 : 2);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                size_t tj = (size_t)t * k + j;
                double v;
                if (cfmt == 1) {
                    int8_t c = ((const int8_t*)(cbuf + tj * rowb))[h];
                    v = (double)c * (double)cscale[tj];
                } else {
                    v = (double)orc_bf16_to_f32(((const uint16_t*)(cbuf + tj * rowb))[h]);
                }
                acc += (double)topk_w[tj] * v;
            }
            out[(size_t)t * H + h] = orc_f64_to_bf16(acc);
        }
    }
    return ORC_OK;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the parallel loops above use from now on (n >= 1); the timed
 * single-thread baseline sets 1.  No effect on any result: every parallel
 * loop writes disjoint rows. */
void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
