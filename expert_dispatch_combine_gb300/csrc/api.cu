// api.cu -- the extern "C" entry points declared in include/moe.h: host-side
// validation, buffer layout, and the launch sequence of each step.
#include <limits.h>
#include <string.h>

#include <atomic>

#include "internal.cuh"

using namespace moe;

namespace moe {
static std::atomic<long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static bool g_prof_on = false;
static cudaEvent_t g_prof_ev[kProfSlots][2] = {};
static bool g_prof_recorded[kProfSlots] = {};
cudaEvent_t prof_event(int slot, int end) {
    if (!g_prof_on) return nullptr;
    if (end) g_prof_recorded[slot] = true;
    return g_prof_ev[slot][end];
}

cudaError_t clear_status(void* ws, cudaStream_t st) {
    count_launches(1);
    return cudaMemsetAsync(ws, 0, 256, st);
}
}  // namespace moe

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bound of each token's wait in moe_expert_ffn_combine (2 s).
constexpr int64_t kCombineWaitNs = 2000000000LL;

moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->T < 1 || s->H < 16 || s->H > 16384 || s->H % 16) return MOE_ERR_INVALID_ARG;
    if (s->I < 16 || s->I > 16384 || s->I % 16) return MOE_ERR_INVALID_ARG;
    if (s->E_log < 1 || s->E_phys < s->E_log || s->E_phys > 1024) return MOE_ERR_INVALID_ARG;
    if (s->k < 1 || s->k > s->E_log || s->k > 32) return MOE_ERR_INVALID_ARG;
    if (s->n_ranks < 1 || s->E_phys % s->n_ranks) return MOE_ERR_INVALID_ARG;
    if (s->n_src_ranks < 1 || s->T % s->n_src_ranks) return MOE_ERR_INVALID_ARG;
    if ((long long)s->T * s->k >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
    if (s->dispatch_fmt != MOE_MSG_BF16 && s->dispatch_fmt != MOE_MSG_INT8) return MOE_ERR_INVALID_ARG;
    if (s->combine_fmt != MOE_MSG_BF16 && s->combine_fmt != MOE_MSG_INT8) return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*s);
    if (d.nslots >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

void fill_layout(const Dims& d, moe_layout* L) {
    L->max_tokens = d.mt;
    L->dispatch_row_bytes = d.drow;
    L->dispatch_meta_offset = align_up(d.nslots * d.drow, 256);
    L->dispatch_bytes = align_up(L->dispatch_meta_offset + d.nslots * (long long)sizeof(moe_dispatch_meta), 256);
    L->combine_row_bytes = d.crow;
    L->combine_scale_offset = align_up((long long)d.T * d.k * d.crow, 256);
    L->combine_bytes = align_up(L->combine_scale_offset + 4LL * d.T * d.k, 256);
    L->workspace_bytes = make_ws(d).total;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    g_last_cuda_error = e;
    return MOE_ERR_CUDA;
}

moe_status check_weights(const Dims& d, const moe_expert_weights* w) {
    if (!w || !w->w_gate_up || !w->s_gate_up || !w->w_down || !w->s_down) return MOE_ERR_INVALID_ARG;
    if (w->n_sets < 1) return MOE_ERR_INVALID_ARG;
    if (!w->phys_to_weight && w->n_sets < d.E_phys) return MOE_ERR_INVALID_ARG;
    if (!aligned(w->w_gate_up, 16) || !aligned(w->w_down, 16)) return MOE_ERR_INVALID_ARG;
    if (!w->w_gate_up_f16 != !w->w_down_f16) return MOE_ERR_INVALID_ARG;  // both or neither
    if (!aligned(w->w_gate_up_f16, 16) || !aligned(w->w_down_f16, 16)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_WORKSPACE: return "buffer or workspace too small";
        case MOE_ERR_CAPACITY: return "static buffer capacity exceeded";
        case MOE_ERR_CUDA: return "CUDA launch error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_INDEX: return "device-side index check failed";
    }
    return "unknown status";
}

moe_status moe_static_buffer_bytes(int64_t rank_num, int64_t local_batch, int64_t topk,
                                   int64_t experts_per_rank, int64_t msg_size, int64_t* bytes) {
    if (!bytes || rank_num < 1 || local_batch < 1 || topk < 1 || experts_per_rank < 1 || msg_size < 1)
        return MOE_ERR_INVALID_ARG;
    const int64_t m = topk < experts_per_rank ? topk : experts_per_rank;
    // rank_num * (local_batch * m) * msg_size without signed overflow
    unsigned __int128 v = (unsigned __int128)rank_num * (unsigned __int128)local_batch;
    v *= (unsigned __int128)m;
    v *= (unsigned __int128)msg_size;
    if (v > (unsigned __int128)INT64_MAX) return MOE_ERR_INVALID_ARG;
    *bytes = (int64_t)v;
    return MOE_OK;
}

moe_status moe_query_layout(const moe_shape* shape, moe_layout* layout) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!layout) return MOE_ERR_INVALID_ARG;
    fill_layout(make_dims(*shape), layout);
    return MOE_OK;
}

moe_status moe_expert_ffn_narrow_rows(const moe_shape* shape, int32_t* rows) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!rows) return MOE_ERR_INVALID_ARG;
    const Dims d = make_dims(*shape);
    const WsLayout wl = make_ws(d);
    *rows = (wl.tc && !ffn_gemv_fits(d)) ? narrow_expert_rows(d) : 0;
    return MOE_OK;
}

moe_status moe_weights_to_f16(const int8_t* src, int64_t n, uint16_t* dst, moe_stream_t stream) {
    if (n < 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;  // nothing to copy; the pointers are not used
    if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_weights_to_f16(src, n, dst, stream));
}

moe_status moe_expert_ffn_path(const moe_shape* shape, int32_t* path) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!path) return MOE_ERR_INVALID_ARG;
    const Dims d = make_dims(*shape);
    const WsLayout wl = make_ws(d);
    *path = !wl.tc ? MOE_FFN_CUDA_CORE : ffn_gemv_fits(d) ? MOE_FFN_GEMV : MOE_FFN_TENSOR_CORE;
    return MOE_OK;
}

moe_status moe_route(const moe_shape* shape, const float* logits, const int32_t* rep_table,
                     const int32_t* n_copies, int32_t max_copies, int32_t* topk_idx,
                     float* topk_w, int32_t* phys_idx, int32_t* expert_counts,
                     moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!logits || !topk_idx || !topk_w || !phys_idx || !expert_counts) return MOE_ERR_INVALID_ARG;
    if (rep_table) {
        if (!n_copies || max_copies < 1) return MOE_ERR_INVALID_ARG;
    } else if (shape->E_phys != shape->E_log) {
        return MOE_ERR_INVALID_ARG;
    }
    Dims d = make_dims(*shape);
    return cuda_status(launch_route(d, logits, rep_table, n_copies, max_copies, topk_idx, topk_w,
                                    phys_idx, expert_counts, (cudaStream_t)stream));
}

moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* phys_idx,
                        void* dispatch_buf, int64_t dispatch_bytes, int32_t* rank_counts,
                        int32_t* expert_offsets, int32_t* expert_rows, void* workspace,
                        int64_t workspace_bytes, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!x || !phys_idx || !dispatch_buf || !rank_counts || !expert_offsets || !expert_rows ||
        !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dispatch_buf, 256) || !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*shape);
    moe_layout L;
    fill_layout(d, &L);
    if (dispatch_bytes < L.dispatch_bytes || workspace_bytes < L.workspace_bytes)
        return MOE_ERR_WORKSPACE;
    return cuda_status(launch_dispatch(d, x, phys_idx, dispatch_buf, L.dispatch_meta_offset,
                                       rank_counts, expert_offsets, expert_rows, workspace,
                                       make_ws(d), (cudaStream_t)stream));
}

moe_status moe_trampoline_bytes(const moe_shape* shape, int64_t* bytes) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!bytes || shape->n_src_ranks > shape->n_ranks) return MOE_ERR_INVALID_ARG;
    *bytes = trampoline_layout(make_dims(*shape)).total;
    return MOE_OK;
}

moe_status moe_dispatch_trampoline(const moe_shape* shape, const uint16_t* x, const int32_t* phys_idx,
                                   void* trampoline_buf, int64_t trampoline_bytes,
                                   void* dispatch_buf, int64_t dispatch_bytes, int32_t* rank_counts,
                                   int32_t* expert_offsets, int32_t* expert_rows, void* workspace,
                                   int64_t workspace_bytes, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->n_src_ranks > shape->n_ranks) return MOE_ERR_INVALID_ARG;
    if (!x || !phys_idx || !trampoline_buf || !dispatch_buf || !rank_counts || !expert_offsets ||
        !expert_rows || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(trampoline_buf, 256) || !aligned(dispatch_buf, 256) ||
        !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*shape);
    moe_layout L;
    fill_layout(d, &L);
    if (dispatch_bytes < L.dispatch_bytes || workspace_bytes < L.workspace_bytes ||
        trampoline_bytes < trampoline_layout(d).total)
        return MOE_ERR_WORKSPACE;
    return cuda_status(launch_dispatch_trampoline(d, x, phys_idx, trampoline_buf, dispatch_buf,
                                                  L.dispatch_meta_offset, rank_counts,
                                                  expert_offsets, expert_rows, workspace,
                                                  make_ws(d), (cudaStream_t)stream));
}

moe_status moe_expert_ffn(const moe_shape* shape, const void* dispatch_buf,
                          int64_t dispatch_bytes, const int32_t* expert_offsets,
                          const int32_t* expert_rows, const moe_expert_weights* weights,
                          void* combine_buf, int64_t combine_bytes, void* workspace,
                          int64_t workspace_bytes, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->dispatch_fmt != MOE_MSG_INT8) return MOE_ERR_UNSUPPORTED;
    if (!dispatch_buf || !expert_offsets || !expert_rows || !combine_buf || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(dispatch_buf, 256) || !aligned(combine_buf, 256) || !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*shape);
    if ((st = check_weights(d, weights)) != MOE_OK) return st;
    moe_layout L;
    fill_layout(d, &L);
    if (dispatch_bytes < L.dispatch_bytes || combine_bytes < L.combine_bytes ||
        workspace_bytes < L.workspace_bytes)
        return MOE_ERR_WORKSPACE;
    return cuda_status(launch_ffn(d, dispatch_buf, L.dispatch_meta_offset, expert_offsets,
                                  expert_rows, *weights, combine_buf, L.combine_scale_offset,
                                  workspace, make_ws(d), (cudaStream_t)stream));
}

moe_status moe_expert_ffn_combine_ex(const moe_shape* shape, const void* dispatch_buf,
                                     int64_t dispatch_bytes, const int32_t* expert_offsets,
                                     const int32_t* expert_rows, const moe_expert_weights* weights,
                                     const float* topk_w, void* combine_buf, int64_t combine_bytes,
                                     uint16_t* out, void* workspace, int64_t workspace_bytes,
                                     int32_t expected, int64_t wait_ns, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->dispatch_fmt != MOE_MSG_INT8) return MOE_ERR_UNSUPPORTED;
    if (!dispatch_buf || !expert_offsets || !expert_rows || !combine_buf || !workspace || !topk_w ||
        !out)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(dispatch_buf, 256) || !aligned(combine_buf, 256) || !aligned(workspace, 256) ||
        !aligned(out, 16))
        return MOE_ERR_INVALID_ARG;
    if (expected < 1 || wait_ns < 1) return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*shape);
    const WsLayout wl = make_ws(d);
    if (!ffn_fuses_combine(d, wl)) return MOE_ERR_UNSUPPORTED;
    if ((st = check_weights(d, weights)) != MOE_OK) return st;
    moe_layout L;
    fill_layout(d, &L);
    if (dispatch_bytes < L.dispatch_bytes || combine_bytes < L.combine_bytes ||
        workspace_bytes < L.workspace_bytes)
        return MOE_ERR_WORKSPACE;
    FusedCombine fc{topk_w, out, expected, (unsigned long long)wait_ns};
    return cuda_status(launch_ffn(d, dispatch_buf, L.dispatch_meta_offset, expert_offsets,
                                  expert_rows, *weights, combine_buf, L.combine_scale_offset,
                                  workspace, wl, (cudaStream_t)stream, fc));
}

moe_status moe_expert_ffn_combine(const moe_shape* shape, const void* dispatch_buf,
                                  int64_t dispatch_bytes, const int32_t* expert_offsets,
                                  const int32_t* expert_rows, const moe_expert_weights* weights,
                                  const float* topk_w, void* combine_buf, int64_t combine_bytes,
                                  uint16_t* out, void* workspace, int64_t workspace_bytes,
                                  moe_stream_t stream) {
    if (!shape) return MOE_ERR_INVALID_ARG;
    return moe_expert_ffn_combine_ex(shape, dispatch_buf, dispatch_bytes, expert_offsets, expert_rows,
                                     weights, topk_w, combine_buf, combine_bytes, out, workspace,
                                     workspace_bytes, shape->k, kCombineWaitNs, stream);
}

moe_status moe_combine(const moe_shape* shape, const void* combine_buf, int64_t combine_bytes,
                       const float* topk_w, uint16_t* out, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!combine_buf || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(combine_buf, 256) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    Dims d = make_dims(*shape);
    moe_layout L;
    fill_layout(d, &L);
    if (combine_bytes < L.combine_bytes) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_combine(d, combine_buf, L.combine_scale_offset, topk_w, out,
                                      (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Host-side checks of moe_layer's arguments (nothing is enqueued).
moe_status check_layer_args(const moe_shape* shape, const float* logits, const uint16_t* x,
                            const int32_t* rep_table, const int32_t* n_copies, int32_t max_copies,
                            const moe_expert_weights* weights, const moe_routing* routing,
                            const void* dispatch_buf, int64_t dispatch_bytes, const void* combine_buf,
                            int64_t combine_bytes, const void* workspace, int64_t workspace_bytes,
                            const uint16_t* out, moe_layout* L) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->dispatch_fmt != MOE_MSG_INT8) return MOE_ERR_UNSUPPORTED;
    if (!routing || !logits || !x || !out) return MOE_ERR_INVALID_ARG;
    const moe_routing& r = *routing;
    if (!r.topk_idx || !r.topk_w || !r.phys_idx || !r.expert_counts || !r.rank_counts ||
        !r.expert_offsets || !r.expert_rows)
        return MOE_ERR_INVALID_ARG;
    if (!dispatch_buf || !combine_buf || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(dispatch_buf, 256) ||
        !aligned(combine_buf, 256) || !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    if (rep_table) {
        if (!n_copies || max_copies < 1) return MOE_ERR_INVALID_ARG;
    } else if (shape->E_phys != shape->E_log) {
        return MOE_ERR_INVALID_ARG;
    }
    Dims d = make_dims(*shape);
    if ((st = check_weights(d, weights)) != MOE_OK) return st;
    fill_layout(d, L);
    if (dispatch_bytes < L->dispatch_bytes || combine_bytes < L->combine_bytes ||
        workspace_bytes < L->workspace_bytes)
        return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_layer(const moe_shape* shape, const float* logits, const uint16_t* x,
                     const int32_t* rep_table, const int32_t* n_copies, int32_t max_copies,
                     const moe_expert_weights* weights, const moe_routing* routing,
                     void* dispatch_buf, int64_t dispatch_bytes, void* combine_buf,
                     int64_t combine_bytes, void* workspace, int64_t workspace_bytes,
                     uint16_t* out, moe_stream_t stream) {
    moe_layout L;
    moe_status st = check_layer_args(shape, logits, x, rep_table, n_copies, max_copies, weights,
                                     routing, dispatch_buf, dispatch_bytes, combine_buf,
                                     combine_bytes, workspace, workspace_bytes, out, &L);
    if (st != MOE_OK) return st;
    const moe_routing& r = *routing;
    const Dims d = make_dims(*shape);
    const WsLayout wl = make_ws(d);
    cudaStream_t s = (cudaStream_t)stream;
    // profiling events around the four steps (slots 4..7), when enabled
    auto mark = [&](int slot, int end) {
        if (cudaEvent_t ev = prof_event(slot, end)) cudaEventRecord(ev, s);
    };
    mark(4, 0);
    if ((st = cuda_status(launch_route(d, logits, rep_table, n_copies, max_copies, r.topk_idx,
                                       r.topk_w, r.phys_idx, r.expert_counts, s))) != MOE_OK)
        return st;
    mark(4, 1);
    // the status word is cleared once, by the dispatch, and covers the whole
    // layer; on the tensor-core FFN path the dispatch also writes the FFN's
    // fp16 input rows, and the FFN skips its assembly step
    const bool stage = ffn_takes_tc(d, wl);
    mark(5, 0);
    if ((st = cuda_status(launch_dispatch(d, x, r.phys_idx, dispatch_buf, L.dispatch_meta_offset,
                                          r.rank_counts, r.expert_offsets, r.expert_rows,
                                          workspace, wl, s, /*clear=*/true, stage))) != MOE_OK)
        return st;
    mark(5, 1);
    mark(6, 0);
    if ((st = cuda_status(launch_ffn(d, dispatch_buf, L.dispatch_meta_offset, r.expert_offsets,
                                     r.expert_rows, *weights, combine_buf, L.combine_scale_offset,
                                     workspace, wl, s, FusedCombine{nullptr, nullptr},
                                     /*clear=*/false, /*rows_ready=*/stage))) != MOE_OK)
        return st;
    mark(6, 1);
    mark(7, 0);
    st = cuda_status(launch_combine(d, combine_buf, L.combine_scale_offset, r.topk_w, out, s));
    mark(7, 1);
    return st;
}

moe_status moe_layer_host(const moe_shape* shape, const float* h_logits, const uint16_t* h_x,
                          uint16_t* h_out, float* d_logits, uint16_t* d_x, const int32_t* rep_table,
                          const int32_t* n_copies, int32_t max_copies,
                          const moe_expert_weights* weights, const moe_routing* routing,
                          void* dispatch_buf, int64_t dispatch_bytes, void* combine_buf,
                          int64_t combine_bytes, void* workspace, int64_t workspace_bytes,
                          uint16_t* d_out, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!h_logits || !h_x || !h_out || !d_logits || !d_x || !d_out) return MOE_ERR_INVALID_ARG;
    if (!aligned(h_logits, 16) || !aligned(h_x, 16) || !aligned(h_out, 16) || !aligned(d_logits, 16))
        return MOE_ERR_INVALID_ARG;
    moe_layout L;
    if ((st = check_layer_args(shape, d_logits, d_x, rep_table, n_copies, max_copies, weights,
                               routing, dispatch_buf, dispatch_bytes, combine_buf, combine_bytes,
                               workspace, workspace_bytes, d_out, &L)) != MOE_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t lg_bytes = sizeof(float) * (size_t)shape->T * shape->E_log;
    const size_t x_bytes = 2 * (size_t)shape->T * shape->H;
    if ((st = cuda_status(cudaMemcpyAsync(d_logits, h_logits, lg_bytes, cudaMemcpyHostToDevice, s))) !=
            MOE_OK ||
        (st = cuda_status(cudaMemcpyAsync(d_x, h_x, x_bytes, cudaMemcpyHostToDevice, s))) != MOE_OK)
        return st;
    count_launches(2);
    if ((st = moe_layer(shape, d_logits, d_x, rep_table, n_copies, max_copies, weights, routing,
                        dispatch_buf, dispatch_bytes, combine_buf, combine_bytes, workspace,
                        workspace_bytes, d_out, stream)) != MOE_OK)
        return st;
    count_launches(1);
    return cuda_status(cudaMemcpyAsync(h_out, d_out, x_bytes, cudaMemcpyDeviceToHost, s));
}

moe_status moe_profile_enable(int32_t on) {
    if (on && !g_prof_on) {
        for (int s = 0; s < kProfSlots; ++s)
            for (int e = 0; e < 2; ++e)
                if (!g_prof_ev[s][e] && cudaEventCreate(&g_prof_ev[s][e]) != cudaSuccess)
                    return cuda_status(cudaGetLastError());
    }
    if (on && !g_prof_on)
        for (int s = 0; s < kProfSlots; ++s) g_prof_recorded[s] = false;
    g_prof_on = on != 0;
    return MOE_OK;
}

moe_status moe_profile_read(float* ms, int32_t n) {
    if (!ms || n < 1) return MOE_ERR_INVALID_ARG;
    for (int s = 0; s < n; ++s) ms[s] = -1.f;
    for (int s = 0; s < kProfSlots && s < n; ++s) {
        if (!g_prof_recorded[s] || !g_prof_ev[s][0] || !g_prof_ev[s][1]) continue;
        if (cudaEventSynchronize(g_prof_ev[s][1]) != cudaSuccess) return cuda_status(cudaGetLastError());
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_prof_ev[s][0], g_prof_ev[s][1]) == cudaSuccess) ms[s] = t;
        else cudaGetLastError();
    }
    return MOE_OK;
}

const char* moe_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

int64_t moe_launch_count(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }

int64_t moe_gemm_workspace_bytes(int32_t n_groups, int64_t max_rows, int32_t K) {
    if (n_groups < 1 || max_rows < 0 || K < 16) return -1;
    return gemm_ws_bytes(n_groups, max_rows, K);
}

moe_status moe_device_status(const void* workspace, int32_t* status, moe_stream_t stream) {
    if (!workspace || !status) return MOE_ERR_INVALID_ARG;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
            cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    *status = v;
    return MOE_OK;
}

moe_status moe_grouped_gemm_s8(int32_t n_groups, const int32_t* offsets, int64_t max_rows,
                               const int32_t* row_index, const int8_t* A, int64_t lda,
                               const int8_t* B, int32_t N, int32_t K, int32_t* C,
                               void* workspace, int64_t workspace_bytes, moe_stream_t stream) {
    if (n_groups < 1 || !offsets || max_rows < 0 || !A || !B || !C || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (K < 16 || K % 16 || K >= (1 << 20) || N < 16 || N % 16 || lda < K || lda % 16)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < gemm_ws_bytes(n_groups, max_rows, K)) return MOE_ERR_WORKSPACE;
    if (max_rows == 0) return MOE_OK;
    if (K % 64 == 0)
        return cuda_status(launch_grouped_gemm_tc(n_groups, offsets, max_rows, row_index, A, lda, B,
                                                  N, K, C, workspace, (cudaStream_t)stream));
    moe_status st = cuda_status(clear_status(workspace, (cudaStream_t)stream));
    if (st != MOE_OK) return st;
    // the rows of A are the caller's: no bound on the row list's entries here
    return cuda_status(launch_grouped_gemm_s8(n_groups, offsets, max_rows, row_index, LLONG_MAX, A,
                                              lda, B, (long long)N * K, nullptr, n_groups, N, K, C,
                                              ws_ptr<int32_t>(workspace, 256),
                                              ws_ptr<int>(workspace, 0), (cudaStream_t)stream));
}

}  // extern "C"

// Status for a CUDA error raised outside this file (records it for
// moe_last_cuda_error like every entry point here).
moe_status moe::record_cuda_status(cudaError_t e) { return cuda_status(e); }
