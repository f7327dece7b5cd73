// Decode-step driver: a layer stack's projections back to back on one stream
// (OpenJet news page, paragraph "并行解码的原理": every projection of every
// layer streams its packed weights once per step).  The launch sequence can be
// captured once into a CUDA graph so a step costs one graph launch on the host.
#include <cuda_runtime.h>

#include <new>

#include "wq.h"

struct wq_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

extern "C" {

wq_status_t wq_step_run(const wq_proj_desc_t* projs, int count, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (count < 0 || (count > 0 && !projs)) return WQ_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const wq_proj_desc_t& p = projs[i];
        wq_status_t st = wq_gemm(p.x, p.wq, p.scales, p.zeros, p.y, p.M, p.N, p.K, p.group, p.bits,
                                 workspace, workspace_bytes, stream);
        if (st != WQ_OK) return st;
    }
    return WQ_OK;
}

wq_status_t wq_step_graph_create(const wq_proj_desc_t* projs, int count, void* workspace,
                                 size_t workspace_bytes, void* stream, wq_step_graph_t* out) {
    if (!out || !workspace || count <= 0 || !projs) return WQ_ERR_INVALID_ARG;
    *out = nullptr;
    // Capture needs a non-legacy stream: use the caller's, or a private one.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t own = nullptr;
    if (s == nullptr) {
        if (cudaStreamCreateWithFlags(&own, cudaStreamNonBlocking) != cudaSuccess) return WQ_ERR_CUDA;
        s = own;
    }
    wq_step_graph* g = new (std::nothrow) wq_step_graph;
    wq_status_t st = g ? WQ_OK : WQ_ERR_CUDA;
    if (st == WQ_OK && cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        st = WQ_ERR_CUDA;
    if (st == WQ_OK) {
        wq_status_t run = wq_step_run(projs, count, workspace, workspace_bytes, s);
        cudaError_t e = cudaStreamEndCapture(s, &g->graph);
        if (run != WQ_OK) st = run;
        else if (e != cudaSuccess) st = WQ_ERR_CUDA;
    }
    if (st == WQ_OK && cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) st = WQ_ERR_CUDA;
    if (own) cudaStreamDestroy(own);
    if (st != WQ_OK) {
        wq_step_graph_destroy(g);
        return st;
    }
    *out = g;
    return WQ_OK;
}

wq_status_t wq_step_graph_launch(wq_step_graph_t g, void* stream) {
    if (!g || !g->exec) return WQ_ERR_INVALID_ARG;
    return cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? WQ_OK
               : WQ_ERR_CUDA;
}

void wq_step_graph_destroy(wq_step_graph_t g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}

}  // extern "C"
