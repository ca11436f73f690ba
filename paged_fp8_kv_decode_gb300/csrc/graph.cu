// graph.cu -- step graphs: the kv_append and attention calls of one decode
// step for a stack of layers, captured once as a CUDA graph and replayed with
// one launch (see pfkv.h).  Host code only; the captured kernels are the ones
// the direct calls launch.
#include <new>

#include "pfkv_internal.cuh"

struct pfkv_step_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    int device;
};

namespace {

pfkv_status cuda_fail() {
    cudaGetLastError();  // clear the error so that later calls start clean
    return PFKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pfkv_status pfkv_step_graph_create(const pfkv_layer *layers, int32_t num_layers,
                                   const pfkv_pages *pages, const int32_t *positions,
                                   const int32_t *new_lens, int32_t num_new_tokens,
                                   uint8_t *append_flags, int32_t num_q_heads, float sm_scale,
                                   int32_t split_tokens, int32_t max_seq_len, void *workspace,
                                   size_t workspace_bytes, uint32_t options,
                                   pfkv_step_graph **graph) {
    if (!graph) return PFKV_ERR_INVALID_ARG;
    *graph = nullptr;
    if (!layers || num_layers <= 0 || !pages) return PFKV_ERR_INVALID_ARG;
    if (options & ~PFKV_STAGE_FUSED_TAGS) return PFKV_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if ((layers[l].k_new == nullptr) != (layers[l].v_new == nullptr)) return PFKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();

    // capture on a private stream, in this thread only
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return cuda_fail();
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(s);
        return cuda_fail();
    }
    pfkv_status st = PFKV_OK;
    for (int l = 0; l < num_layers && st == PFKV_OK; ++l) {
        const pfkv_layer &L = layers[l];
        if (L.k_new)  // append + attention as one step (append and validation share a launch)
            st = pfkv_decode_step(&L.cache, pages, positions, new_lens, num_new_tokens, L.k_new, L.v_new,
                                  append_flags, L.q, num_q_heads, sm_scale, split_tokens, max_seq_len,
                                  workspace, workspace_bytes, L.out, L.flags, options, s);
        else
            st = pfkv_paged_decode_attn_stages(&L.cache, pages, L.q, num_q_heads, sm_scale,
                                               split_tokens, max_seq_len, workspace, workspace_bytes,
                                               L.out, L.flags, PFKV_STAGE_ALL | options, s);
    }
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(s, &g);
    cudaStreamDestroy(s);
    if (st != PFKV_OK || ce != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return st != PFKV_OK ? st : PFKV_ERR_CUDA;
    }
    cudaGraphExec_t x = nullptr;
    if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        return cuda_fail();
    }
    pfkv_step_graph *h = new (std::nothrow) pfkv_step_graph{g, x, dev};
    if (!h) {
        cudaGraphExecDestroy(x);
        cudaGraphDestroy(g);
        return PFKV_ERR_CUDA;
    }
    *graph = h;
    return PFKV_OK;
}

pfkv_status pfkv_step_graph_launch(pfkv_step_graph *graph, void *stream) {
    if (!graph) return PFKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    if (dev != graph->device) return PFKV_ERR_INVALID_ARG;  // made on another device
    if (cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_fail();
    return PFKV_OK;
}

pfkv_status pfkv_step_graph_destroy(pfkv_step_graph *graph) {
    if (!graph) return PFKV_OK;
    const bool ok = cudaGraphExecDestroy(graph->exec) == cudaSuccess &&
                    cudaGraphDestroy(graph->graph) == cudaSuccess;
    delete graph;
    if (!ok) return cuda_fail();
    return PFKV_OK;
}

}  // extern "C"
