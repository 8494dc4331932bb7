// CUDA graphs of the decode step: one capture of llama_stack_decode, replayed step after step.
//
// A decode step of a deep stack is hundreds of short kernels ("第 10 章：现代 LLaMA 架构" §7:
// one token per sequence through every layer); replaying them as one graph removes the
// per-launch host cost and keeps the programmatic-dependent-launch edges between them.
// The captured arguments are pointers, so the caller drives the next step by writing the
// new tokens and positions into the same device buffers before each replay.
#include <cuda_runtime.h>

#include "internal.h"

struct llama_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  int device;
  int kernels;
};

extern "C" {

int llama_stack_decode_graph(const llama_stack* st, const int32_t* tokens, const int32_t* positions, float* logits,
                             const float* cos, const float* sin, int32_t max_pos, const llama_kv_cache* caches,
                             int32_t B, void* workspace, size_t ws_bytes, llama_graph** out) {
  using namespace llama;
  if (out == nullptr) return LLAMA_ERR_INVALID_ARG;
  *out = nullptr;
  if (trace_active()) return LLAMA_ERR_INVALID_ARG;   // trace events must not end up in the graph
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return LLAMA_ERR_CUDA;
  // capture on a private stream, so that nothing else the caller has queued is recorded
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return LLAMA_ERR_CUDA;
  const uint64_t before = llama_kernel_launch_count();
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(s);
    return LLAMA_ERR_CUDA;
  }
  int rc = llama_stack_decode(st, tokens, positions, logits, cos, sin, max_pos, caches, B, workspace, ws_bytes, s);
  cudaGraph_t g = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &g);   // ends the capture whatever happened above
  const int kernels = static_cast<int>(llama_kernel_launch_count() - before);
  cudaStreamDestroy(s);
  if (rc == LLAMA_OK && (end != cudaSuccess || g == nullptr)) rc = LLAMA_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == LLAMA_OK && cudaGraphInstantiateWithFlags(&exec, g, 0) != cudaSuccess) rc = LLAMA_ERR_CUDA;
  if (rc != LLAMA_OK) {
    if (g != nullptr) cudaGraphDestroy(g);
    cudaGetLastError();   // clear a capture error so that it does not surface in a later call
    return rc;
  }
  *out = new llama_graph{g, exec, device, kernels};
  return LLAMA_OK;
}

int llama_graph_launch(llama_graph* graph, void* cuda_stream) {
  if (graph == nullptr) return LLAMA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (device != graph->device) return LLAMA_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? LLAMA_OK
                                                                                               : LLAMA_ERR_CUDA;
}

int32_t llama_graph_kernel_count(const llama_graph* graph) { return graph == nullptr ? -1 : graph->kernels; }

int llama_graph_destroy(llama_graph* graph) {
  if (graph == nullptr) return LLAMA_OK;
  const bool ok = cudaGraphExecDestroy(graph->exec) == cudaSuccess && cudaGraphDestroy(graph->graph) == cudaSuccess;
  delete graph;
  return ok ? LLAMA_OK : LLAMA_ERR_CUDA;
}

}  // extern "C"
