// graph.cu -- a whole device-resident prefill captured once into a CUDA graph
// and replayed with one launch.
//
// A prefill of a short sequence is a handful of small kernels (quantise K and
// V, state init, one chunk step per KV chunk, finalise: "Out-of-Core Flash
// Streaming & Speculative Decode (1M Context)", §3 steps 1-6 and the final
// division, chunk by chunk).  Launched one by one from the host, the device
// waits on the host between them; replayed from a graph, the kernels follow one
// another on the device.  The graph holds exactly the launches the calls would
// make, with the arguments they had at capture time.  Host code only.

#include <cstdio>
#include <new>

#include "../../include/q8attn.h"
#include "internal.h"

struct q8a_prefill_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

namespace {

constexpr const char* kCreate = "q8a_prefill_graph_create";

int cuda_err(cudaError_t e, const char* fn, const char* what) {
  char msg[256];
  std::snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorName(e));
  return q8a::set_error(Q8A_ERR_CUDA, fn, msg);
}

// The prefill's launches, in the order the device-resident path makes them.
int enqueue_prefill(const void* q, const float* k, const float* v, void* k8, void* v8,
                    int64_t plane_stride_bytes, float* m, float* l, float* o, void* out,
                    int64_t batch, int32_t heads, int64_t n_tokens, int32_t head_dim, int64_t chunk,
                    float scale, int32_t causal, void* stream) {
  int rc;
  if ((rc = q8kv_quantize(k, k8, batch, n_tokens, heads, head_dim, plane_stride_bytes, stream)) != Q8A_OK ||
      (rc = q8kv_quantize(v, v8, batch, n_tokens, heads, head_dim, plane_stride_bytes, stream)) != Q8A_OK ||
      (rc = attn_state_init(m, l, o, batch, heads, n_tokens, head_dim, stream)) != Q8A_OK)
    return rc;
  const int64_t row_bytes = head_dim / 32 * 34;
  for (int64_t s0 = 0; s0 < n_tokens; s0 += chunk) {
    const int64_t n = (n_tokens - s0 < chunk) ? n_tokens - s0 : chunk;
    const uint8_t* kc = static_cast<const uint8_t*>(k8) + s0 * row_bytes;
    const uint8_t* vc = static_cast<const uint8_t*>(v8) + s0 * row_bytes;
    if ((rc = attn_chunk_step(q, 0, kc, vc, plane_stride_bytes, s0, n, m, l, o, batch, heads, n_tokens,
                              head_dim, scale, causal, stream)) != Q8A_OK)
      return rc;
  }
  return attn_finalize(l, o, out, batch, heads, n_tokens, head_dim, stream);
}

}  // namespace

extern "C" {

int q8a_prefill_graph_create(const void* q, const float* k, const float* v, void* k8, void* v8,
                             int64_t plane_stride_bytes, float* m, float* l, float* o, void* out,
                             int64_t batch, int32_t heads, int64_t n_tokens, int32_t head_dim,
                             int64_t chunk, float scale, int32_t causal, q8a_prefill_graph** graph_out) {
  q8a::NvtxRange nvtx_range(kCreate);
  if (!graph_out) return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate, "graph_out is null");
  *graph_out = nullptr;
  if (batch < 0 || heads <= 0 || n_tokens < 0 || chunk <= 0)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate, "sizes must be >= 0, heads and chunk > 0");
  if (head_dim != 64 && head_dim != 128)
    return q8a::set_error(Q8A_ERR_UNSUPPORTED, kCreate, "head_dim must be 64 or 128");
  // every chunk start must leave the chunk's Q8_0 rows 16-byte aligned
  if (chunk % (head_dim == 64 ? 4 : 2) != 0)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate,
                          "chunk must be a multiple of 4 (head_dim 64) or 2 (head_dim 128)");
  if (!q || !k || !v || !k8 || !v8 || !m || !l || !o || !out)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate, "null pointer");
  if (!(scale > 0.0f))
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate, "scale must be > 0");
  const int64_t min_stride = q8a_plane_stride_bytes_for(n_tokens, head_dim);
  if (plane_stride_bytes < min_stride || plane_stride_bytes % 16 != 0)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kCreate,
                          "plane_stride_bytes must be >= n_tokens*head_dim/32*34 and a multiple of 16");

  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_err(e, kCreate, "cudaGetDevice");
  // captured on a private stream, so that no other work joins the graph
  cudaStream_t cs = nullptr;
  if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess)
    return cuda_err(e, kCreate, "cudaStreamCreateWithFlags");
  if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_err(e, kCreate, "cudaStreamBeginCapture");
  }
  int rc;
  {
    // consecutive kernels of the graph with programmatic dependencies: each
    // may be scheduled while its predecessor's last CTAs run, and waits for
    // the predecessor's completion before it touches memory
    q8a::PdlScope pdl;
    rc = enqueue_prefill(q, k, v, k8, v8, plane_stride_bytes, m, l, o, out, batch, heads, n_tokens, head_dim,
                         chunk, scale, causal, cs);
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (rc != Q8A_OK) {   // the failing call's message stays the thread's last error
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return cuda_err(e, kCreate, "cudaStreamEndCapture");
  }
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaGraphInstantiate(&exec, graph, 0)) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_err(e, kCreate, "cudaGraphInstantiate");
  }
  q8a_prefill_graph* g = new (std::nothrow) q8a_prefill_graph;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return q8a::set_error(Q8A_ERR_CUDA, kCreate, "out of host memory for the graph handle");
  }
  g->graph = graph;
  g->exec = exec;
  g->device = device;
  *graph_out = g;
  return q8a::clear_error();
}

int q8a_prefill_graph_launch(q8a_prefill_graph* graph, void* stream) {
  constexpr const char* kFn = "q8a_prefill_graph_launch";
  q8a::NvtxRange nvtx_range(kFn);
  if (!graph || !graph->exec) return q8a::set_error(Q8A_ERR_INVALID_ARG, kFn, "graph is null");
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_err(e, kFn, "cudaGetDevice");
  if (device != graph->device)
    return q8a::set_error(Q8A_ERR_INVALID_ARG, kFn, "the current device is not the graph's device");
  if ((e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_err(e, kFn, "cudaGraphLaunch");
  return q8a::clear_error();
}

int q8a_prefill_graph_destroy(q8a_prefill_graph* graph) {
  if (!graph) return Q8A_OK;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
  return Q8A_OK;
}

}  // extern "C"
