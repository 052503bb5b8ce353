// graph.cu -- the decode layer as a CUDA graph.
//
// "CloudMatrix384 LLM Serving", section "EP320：token 去找专家": the static
// dispatch/combine buffers are allocated once and reused by every decode
// step, and they are double-buffered so that one step's combine cannot
// overwrite dispatch data another step still uses.  With buffers that never
// move, one moe_layer call can be captured once and replayed each step: the
// graph reads whatever the captured logits and x buffers hold at launch.
// Double buffering is two graphs over two buffer sets, replayed in turn.
#include <new>

#include "internal.cuh"

struct moe_graph_s {
    cudaGraphExec_t exec;
};

extern "C" moe_status moe_layer_graph_create(
    const moe_shape* shape, const float* logits, const uint16_t* x, const int32_t* rep_table,
    const int32_t* n_copies, int32_t max_copies, const moe_expert_weights* weights,
    const moe_routing* routing, void* dispatch_buf, int64_t dispatch_bytes, void* combine_buf,
    int64_t combine_bytes, void* workspace, int64_t workspace_bytes, uint16_t* out,
    moe_stream_t capture_stream, moe_graph* graph) {
    if (!graph) return MOE_ERR_INVALID_ARG;
    *graph = nullptr;
    // the legacy default stream cannot be captured
    if (!capture_stream) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)capture_stream;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return moe::record_cuda_status(e);
    if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_INVALID_ARG;
    if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
        return moe::record_cuda_status(e);
    const moe_status st = moe_layer(shape, logits, x, rep_table, n_copies, max_copies, weights,
                                    routing, dispatch_buf, dispatch_bytes, combine_buf,
                                    combine_bytes, workspace, workspace_bytes, out, capture_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t ee = cudaStreamEndCapture(s, &g);  // always ends the capture
    if (st != MOE_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
    }
    if (ee != cudaSuccess || !g) return moe::record_cuda_status(ee != cudaSuccess ? ee : cudaErrorUnknown);
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) return moe::record_cuda_status(ie);
    moe_graph h = new (std::nothrow) moe_graph_s{exec};
    if (!h) {
        cudaGraphExecDestroy(exec);
        return MOE_ERR_CUDA;
    }
    *graph = h;
    return MOE_OK;
}

extern "C" moe_status moe_graph_launch(moe_graph graph, moe_stream_t stream) {
    if (!graph) return MOE_ERR_INVALID_ARG;
    return moe::record_cuda_status(cudaGraphLaunch(graph->exec, (cudaStream_t)stream));
}

extern "C" moe_status moe_graph_destroy(moe_graph graph) {
    if (!graph) return MOE_OK;
    const cudaError_t e = cudaGraphExecDestroy(graph->exec);
    delete graph;
    return moe::record_cuda_status(e);
}
