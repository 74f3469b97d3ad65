// pa_graph.cu -- one serving step (block copies, slot scatter, attention)
// captured into a CUDA graph over fixed, caller-owned buffers.
//
// The continuous-batching pages ("PagedAttention 显存分页与连续批处理
// (Continuous Batching)实战", continuous batching and Chunked Prefill
// sections) run the same operations every step over a different set of
// requests.  Sized for the largest step and padded, that sequence is a fixed
// graph: one launch replaces the three to five kernel launches of the step
// and the per-step metadata can ride in with one host-to-device copy node.
// The captured calls are the library's own public entry points, so the graph
// checks and computes exactly what those calls do; a graph whose steps have
// decode rows only (max_q_len 1) runs scatter + attention as pa_decode_step,
// one with prefill rows runs pa_reshape_and_cache, then pa_paged_attention.
#include <cuda_runtime.h>

#include <new>

#include "pagedattn.h"
#include "pa_internal.h"

struct pa_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

namespace {

int graph_fail(cudaError_t e, const char* what) {
  return pa::api_fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                      cudaGetErrorString(e));
}

// The step's operations, in order, on `s` (which is being captured).
int record_step(const pa_step_buffers& b, cudaStream_t s) {
  if (b.host_meta) {
    cudaError_t e = cudaMemcpyAsync(b.dev_meta, b.host_meta, b.meta_bytes,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return graph_fail(e, "step metadata copy");
  }
  int st = PA_OK;
  if (b.max_pairs > 0) {
    st = pa_copy_blocks(b.k_cache, b.v_cache, b.num_blocks, b.block_size, b.num_kv_heads,
                        b.head_dim, b.copy_pairs, b.max_pairs, s);
    if (st) return st;
  }
  if (b.max_q_len <= 1) {
    // decode rows only: scatter and attention in one kernel
    st = pa_decode_step(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.num_blocks, b.block_size,
                        b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_tables, b.max_blocks,
                        b.seq_lens, b.query_start_loc, b.max_seqs, b.max_tokens, b.max_seq_len,
                        b.slot_mapping, b.scale, b.out, b.workspace, b.workspace_bytes, s);
    if (st) return st;
  } else {
    // mixed rows: scatter, then attention.  (pa_paged_attention_step does
    // both in the attention kernels, but every later query tile of a chunk
    // then reads the chunk's new rows from k_new / v_new instead of the
    // cache, and on the chunked-prefill step and the serving trace that
    // measured slower than one scatter launch.)
    st = pa_reshape_and_cache(b.k_new, b.v_new, b.max_tokens, b.k_cache, b.v_cache, b.num_blocks,
                              b.block_size, b.num_kv_heads, b.head_dim, b.slot_mapping, s);
    if (st) return st;
    st = pa_paged_attention(b.q, b.k_cache, b.v_cache, b.num_blocks, b.block_size, b.num_q_heads,
                            b.num_kv_heads, b.head_dim, b.block_tables, b.max_blocks, b.seq_lens,
                            b.query_start_loc, b.max_seqs, b.max_tokens, b.max_q_len,
                            b.max_seq_len, b.scale, b.out, b.workspace, b.workspace_bytes, s);
    if (st) return st;
  }
  if (b.host_out) {
    cudaError_t e = cudaMemcpyAsync(b.host_out, b.out, b.out_copy_bytes, cudaMemcpyDeviceToHost,
                                    s);
    if (e != cudaSuccess) return graph_fail(e, "step output copy");
  }
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_step_graph_create(const pa_step_buffers* b, pa_step_graph** out) {
  if (!b || !out) return pa::api_fail(PA_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (b->max_tokens <= 0 || b->max_seqs <= 0 || b->max_blocks <= 0 || b->max_pairs < 0 ||
      b->max_q_len <= 0 || b->max_seq_len <= 0)
    return pa::api_fail(PA_ERR_INVALID_ARG,
                        "step maxima must be positive (max_pairs may be 0): tokens %d seqs %d "
                        "blocks %d pairs %d q_len %d seq_len %d",
                        b->max_tokens, b->max_seqs, b->max_blocks, b->max_pairs, b->max_q_len,
                        b->max_seq_len);
  if (b->max_pairs > 0 && !b->copy_pairs)
    return pa::api_fail(PA_ERR_INVALID_ARG, "copy_pairs is NULL with max_pairs %d",
                        b->max_pairs);
  if (b->host_meta && (!b->dev_meta || b->meta_bytes == 0))
    return pa::api_fail(PA_ERR_INVALID_ARG, "host_meta needs dev_meta and meta_bytes");
  if (b->host_out && (b->out_copy_bytes == 0 ||
                      b->out_copy_bytes > (size_t)b->max_tokens * b->num_q_heads * b->head_dim *
                                              sizeof(pa_bf16)))
    return pa::api_fail(PA_ERR_INVALID_ARG, "out_copy_bytes %zu outside (0, out's size]",
                        b->out_copy_bytes);
  // Look up the per-device state outside the capture.
  int st = pa::api_warm_device();
  if (st) return st;

  pa_step_graph* g = new (std::nothrow) pa_step_graph;
  if (!g) return pa::api_fail(PA_ERR_CUDA, "out of host memory");
  cudaGetDevice(&g->device);
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    delete g;
    return graph_fail(e, "cudaStreamCreate");
  }
  // Relaxed: the launchers may set a kernel attribute on first use.
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(s);
    delete g;
    return graph_fail(e, "cudaStreamBeginCapture");
  }
  st = record_step(*b, s);
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(s, &graph);  // always end the capture, even after a failure
  cudaStreamDestroy(s);
  if (st || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    delete g;
    return st ? st : graph_fail(e, "cudaStreamEndCapture");
  }
  e = cudaGraphInstantiate(&g->exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    delete g;
    return graph_fail(e, "cudaGraphInstantiate");
  }
  g->graph = graph;
  *out = g;
  return PA_OK;
}

int pa_step_graph_launch(pa_step_graph* g, cudaStream_t stream) {
  if (!g || !g->exec) return pa::api_fail(PA_ERR_INVALID_ARG, "null graph");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != g->device)
    return pa::api_fail(PA_ERR_INVALID_ARG, "graph was built on device %d, current is %d",
                        g->device, dev);
  pa::NvtxRange range("pa_step_graph_launch");
  cudaError_t e = cudaGraphLaunch(g->exec, stream);
  if (e != cudaSuccess) return graph_fail(e, "cudaGraphLaunch");
  return PA_OK;
}

int pa_step_graph_destroy(pa_step_graph* g) {
  if (!g) return PA_OK;
  cudaError_t e1 = g->exec ? cudaGraphExecDestroy(g->exec) : cudaSuccess;
  cudaError_t e2 = g->graph ? cudaGraphDestroy(g->graph) : cudaSuccess;
  delete g;
  if (e1 != cudaSuccess) return graph_fail(e1, "cudaGraphExecDestroy");
  if (e2 != cudaSuccess) return graph_fail(e2, "cudaGraphDestroy");
  return PA_OK;
}

}  // extern "C"
