// Decode steps replayed as one CUDA graph.
//
// At small batch a decode step is a chain of short kernels and the GPU waits
// on the host between launches (the closing remark of "S12 FlashAttention":
// the kernel is efficient, but the GPU spends its time waiting for the CPU).
// fa_decode_graph_create records the paged decodes of one step -- one call per
// layer, each with its own query, caches and outputs, all sharing the block
// table, the sequence lengths and the split workspace -- into a CUDA graph;
// fa_decode_graph_launch replays them with a single host call.  The graph holds
// the device pointers it was built with: between launches the caller rewrites
// the buffers' contents (new queries, appended keys, longer seq_lens), not the
// pointers.
#include <cuda_runtime.h>

#include <new>

#include "fa_internal.h"

struct fa_decode_graph {
  cudaGraphExec_t exec = nullptr;
  int num_calls = 0;
  int launches_per_call = 0;
};

extern "C" {

int fa_decode_graph_create(fa_decode_graph** graph, int num_calls, const void* const* q, const void* const* k_cache,
                           const void* const* v_cache, void* const* o, float* const* lse,
                           const int32_t* block_table, const int32_t* seq_lens, int B, int Hq, int Hkv, int d,
                           int block_size, int max_blocks, int num_blocks, int num_splits, float scale,
                           void* workspace, size_t ws_bytes) {
  if (graph == nullptr) return FA_ERR_INVALID_ARG;
  *graph = nullptr;
  if (num_calls < 1 || q == nullptr || k_cache == nullptr || v_cache == nullptr || o == nullptr)
    return FA_ERR_INVALID_ARG;
  // everything that must not happen inside a capture: symbol lookup, kernel
  // attributes, the tensor-map encoder
  if (fa::device_status_ptr() == nullptr || fa::decode_prepare() != FA_OK || !fa::encode_init()) return FA_ERR_CUDA;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
  int st = FA_OK;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    return FA_ERR_CUDA;
  }
  for (int i = 0; i < num_calls && st == FA_OK; ++i)
    st = fa_paged_decode(q[i], k_cache[i], v_cache[i], block_table, seq_lens, o[i], lse ? lse[i] : nullptr, B, Hq,
                         Hkv, d, block_size, max_blocks, num_blocks, num_splits, scale, workspace, ws_bytes, s);
  const cudaError_t end = cudaStreamEndCapture(s, &g);  // always ends the capture
  if (st == FA_OK && end != cudaSuccess) st = FA_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (st == FA_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) st = FA_ERR_CUDA;
  if (g != nullptr) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  if (st != FA_OK) {
    if (exec != nullptr) cudaGraphExecDestroy(exec);
    cudaGetLastError();  // a failed capture leaves no sticky error behind
    return st;
  }
  fa_decode_graph* h = new (std::nothrow) fa_decode_graph;
  if (h == nullptr) {
    cudaGraphExecDestroy(exec);
    return FA_ERR_CUDA;
  }
  h->exec = exec;
  h->num_calls = num_calls;
  h->launches_per_call = (num_splits == 1) ? 1 : 2;
  *graph = h;
  return FA_OK;
}

int fa_decode_graph_launch(fa_decode_graph* graph, void* stream) {
  if (graph == nullptr || graph->exec == nullptr) return FA_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_decode_graph_kernel_count(const fa_decode_graph* graph) {
  return graph == nullptr ? 0 : graph->num_calls * graph->launches_per_call;
}

void fa_decode_graph_destroy(fa_decode_graph* graph) {
  if (graph == nullptr) return;
  if (graph->exec != nullptr) cudaGraphExecDestroy(graph->exec);
  delete graph;
}

}  // extern "C"
