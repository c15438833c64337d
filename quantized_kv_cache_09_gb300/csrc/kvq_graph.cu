// kvq_graph.cu -- decode steps (append of the new tokens + decode attention,
// one per layer or per step) captured into one CUDA graph and replayed.  CUDA
// Graph instance reuse, "hardware-aware scheduling" (jsqmd.com/news/887038)
// section 4.1: the graph is captured once and later bound to other tensor
// addresses with cudaGraphExecUpdate instead of being rebuilt.  Host code
// only: the graph holds the same kernel launches the eager calls make, with
// the same programmatic-dependent-launch edges between consecutive launches.
#include <cuda_runtime.h>

#include <new>

#include "kvq.h"
#include "kvq_internal.h"

struct kvq_step_graph {
    cudaGraphExec_t exec;
};

namespace {

// Capture the steps into a new (not instantiated) graph.  The arguments are
// checked by the calls themselves before they launch anything, so a rejected
// step ends the capture with the calls' own status.
kvq_status capture_steps(const kvq_cache *caches, const kvq_step_args *args, int32_t n, cudaGraph_t *graph_out)
{
    *graph_out = nullptr;
    if (!caches || !args || n < 1) return KVQ_ERR_INVALID_ARG;
    // Occupancy queries and function attributes are resolved (and cached)
    // outside the capture: they are not stream work.
    for (int32_t i = 0; i < n; i++) {
        const kvq_cache *c = &caches[i];
        const kvq_step_args *a = &args[i];
        if (c->num_heads > 0 && a->num_q_heads > 0 && a->num_q_heads % c->num_heads == 0 &&
            kvq_decode_workspace_bytes_gqa(static_cast<kvq_format>(c->fmt), c->num_heads, a->num_q_heads,
                                           kvq::kHeadDim) > 0 &&
            kvq::decode_prepare(c->fmt, a->num_q_heads / c->num_heads) < 1)
            return KVQ_ERR_CUDA;
    }
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(s);
        return KVQ_ERR_CUDA;
    }
    const kvq_stream_t ks = reinterpret_cast<kvq_stream_t>(s);
    kvq_status st = KVQ_OK;
    for (int32_t i = 0; i < n && st == KVQ_OK; i++) {
        const kvq_cache *c = &caches[i];
        const kvq_step_args *a = &args[i];
        st = kvq_append(c, a->k_new, a->v_new, a->cu_seqlens, a->block_table, a->max_blocks_per_seq,
                        a->seq_lens_before, a->num_seqs, a->total_new_tokens, a->max_new_tokens, ks);
        if (st == KVQ_OK)
            st = kvq_decode_attention_gqa(c, a->q, a->num_q_heads, a->block_table, a->max_blocks_per_seq,
                                          a->seq_lens, a->num_seqs, a->softmax_scale, a->out, a->workspace,
                                          a->workspace_bytes, ks);
    }
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &g);
    cudaStreamDestroy(s);
    if (st != KVQ_OK || e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return st != KVQ_OK ? st : KVQ_ERR_CUDA;
    }
    *graph_out = g;
    return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_step_graph_create(const kvq_cache *caches, const kvq_step_args *args, int32_t num_steps,
                                 kvq_step_graph **graph_out)
{
    if (!graph_out) return KVQ_ERR_INVALID_ARG;
    *graph_out = nullptr;
    cudaGraph_t g;
    const kvq_status st = capture_steps(caches, args, num_steps, &g);
    if (st != KVQ_OK) return st;
    cudaGraphExec_t exec;
    const cudaError_t e = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    kvq_step_graph *h = new (std::nothrow) kvq_step_graph{exec};
    if (!h) {
        cudaGraphExecDestroy(exec);
        return KVQ_ERR_CUDA;
    }
    *graph_out = h;
    return KVQ_OK;
}

kvq_status kvq_step_graph_update(kvq_step_graph *graph, const kvq_cache *caches, const kvq_step_args *args,
                                 int32_t num_steps)
{
    if (!graph) return KVQ_ERR_INVALID_ARG;
    cudaGraph_t g;
    const kvq_status st = capture_steps(caches, args, num_steps, &g);
    if (st != KVQ_OK) return st;
    cudaGraphExecUpdateResultInfo info;
    cudaError_t e = cudaGraphExecUpdate(graph->exec, g, &info);
    if (e != cudaSuccess) {  // another launch structure: the executable graph is unchanged; build a new one
        (void)cudaGetLastError();
        cudaGraphExec_t exec;
        e = cudaGraphInstantiate(&exec, g, 0);
        if (e == cudaSuccess) {
            cudaGraphExecDestroy(graph->exec);
            graph->exec = exec;
        }
    }
    cudaGraphDestroy(g);
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_step_graph_launch(const kvq_step_graph *graph, kvq_stream_t stream)
{
    if (!graph) return KVQ_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK
                                                                                              : KVQ_ERR_CUDA;
}

kvq_status kvq_step_graph_destroy(kvq_step_graph *graph)
{
    if (!graph) return KVQ_OK;
    const cudaError_t e = cudaGraphExecDestroy(graph->exec);
    delete graph;
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // extern "C"
