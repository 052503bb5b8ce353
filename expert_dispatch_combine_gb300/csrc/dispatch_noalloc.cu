// dispatch_noalloc.cu -- FusedDispatch for callers that cannot provide a
// workspace.
//
// Some callers cannot call cudaMalloc at all:
//   - a serving engine whose allocator has already reserved all device memory
//     and forbids any allocation outside its pool;
//   - a latency-critical decode loop that must not risk the device-wide
//     synchronisation an allocation or free can bring;
//   - a plug-in loaded into a host process that owns all device memory
//     decisions.
// For them, moe_dispatch_noalloc runs the same dispatch kernels as
// moe_dispatch, but its scratch (per-message slot and rank arrays and the
// per-source histograms) lives in a fixed device array of this file rather
// than in a caller-provided workspace.  The caller still passes every input
// and output buffer.
//
// The array, kNoallocScratchBytes (4 MiB), is a file-scope __device__
// variable: every GPU that loads this library holds it until the process
// exits.  Shapes whose scratch does not fit are rejected with
// MOE_ERR_WORKSPACE before anything is enqueued.  Every call shares the
// array; its contents are those of the last call (the dispatch kernels write
// every scratch word they later read; the status word at its start, where
// the device-side index checks post their codes, is cleared by each call
// and not exposed), and calls that overlap on the GPU -- on different
// streams, or from several host threads -- race on it.
#include <mutex>

#include "internal.cuh"

namespace {

constexpr long long kNoallocScratchBytes = 4LL << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the variable's name is only a host-side
// stand-in; its device address must come from cudaGetSymbolAddress.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int64_t moe_dispatch_noalloc_max_scratch(void) { return kNoallocScratchBytes; }

extern "C" moe_status moe_dispatch_noalloc(const moe_shape* shape, const uint16_t* x,
                                           const int32_t* phys_idx, void* dispatch_buf,
                                           int64_t dispatch_bytes, int32_t* rank_counts,
                                           int32_t* expert_offsets, int32_t* expert_rows,
                                           moe_stream_t stream) {
    moe_layout L;
    moe_status st = moe_query_layout(shape, &L);  // validates the shape
    if (st != MOE_OK) return st;
    if (!x || !phys_idx || !dispatch_buf || !rank_counts || !expert_offsets || !expert_rows)
        return MOE_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(dispatch_buf, 256)) return MOE_ERR_INVALID_ARG;
    if (dispatch_bytes < L.dispatch_bytes) return MOE_ERR_WORKSPACE;
    const moe::Dims d = moe::make_dims(*shape);
    const moe::WsLayout wl = moe::make_ws(d);
    // the dispatch kernels use the workspace only below the tile-prefix region
    if (wl.tiles > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;
    void* scratch = nullptr;
    const cudaError_t es = scratch_for_current_device(&scratch);
    if (es != cudaSuccess) return moe::record_cuda_status(es);
    return moe::record_cuda_status(moe::launch_dispatch(d, x, phys_idx, dispatch_buf,
                                                        L.dispatch_meta_offset, rank_counts,
                                                        expert_offsets, expert_rows, scratch, wl,
                                                        (cudaStream_t)stream));
}
