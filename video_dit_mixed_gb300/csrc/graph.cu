// Data-dependent branches inside a captured CUDA graph.
//
// One denoising step of a DiT runs, per block, exactly one of four bodies
// (NVFP4, INT8, BF16 compute, or the TDC skip) chosen on the device by the
// policy kernel.  Instead of launching every kernel and letting the ones of
// the other modes return at once, a step is captured once with a SWITCH
// conditional node per block: a one-thread selector kernel reads the mode
// word and sets the node's condition, and only the chosen body's kernels run
// when the graph is replayed.
#include <cstdint>
#include <new>

#include "common.cuh"
#include "internal.h"

struct sixbit_switch {
  cudaStream_t body_stream;
  cudaGraph_t bodies[8];
  int n;
  int open_branch;
};

namespace sixbit {

__global__ void switch_select_kernel(cudaGraphConditionalHandle h, const int32_t* mode_dev, int first_mode,
                                     unsigned int none) {
  if (threadIdx.x != 0) return;
  const int v = SIXBIT_MODE_OF(*mode_dev) - first_mode;
  cudaGraphSetConditional(h, (v >= 0 && static_cast<unsigned int>(v) < none) ? static_cast<unsigned int>(v) : none);
}

}  // namespace sixbit

using namespace sixbit;

static sixbit_status add_switch_node(cudaStream_t st, cudaStream_t body_stream, cudaGraphConditionalHandle handle,
                                     int nbranches, sixbit_switch** out);

extern "C" sixbit_status sixbit_graph_switch_begin(void* stream, void* body_stream, const int32_t* mode_dev,
                                                   int first_mode, int nbranches, sixbit_switch** out) {
  if (stream == nullptr || body_stream == nullptr || body_stream == stream || mode_dev == nullptr ||
      out == nullptr || nbranches < 1 || nbranches > 8)
    return SIXBIT_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus status;
  cudaGraph_t graph = nullptr;
  if (cudaStreamGetCaptureInfo(st, &status, nullptr, &graph) != cudaSuccess) return SIXBIT_ECUDA;
  if (status != cudaStreamCaptureStatusActive || graph == nullptr) return SIXBIT_EINVAL;

  // a missing selection (default value) runs no body
  cudaGraphConditionalHandle handle;
  if (cudaGraphConditionalHandleCreate(&handle, graph, static_cast<unsigned int>(nbranches),
                                       cudaGraphCondAssignDefault) != cudaSuccess)
    return SIXBIT_ECUDA;
  switch_select_kernel<<<1, 32, 0, st>>>(handle, mode_dev, first_mode, static_cast<unsigned int>(nbranches));
  note_launch();
  if (cudaGetLastError() != cudaSuccess) return SIXBIT_ECUDA;
  return add_switch_node(st, static_cast<cudaStream_t>(body_stream), handle, nbranches, out);
}

// Appends a SWITCH node on `handle` with `nbranches` empty bodies after the
// current capture dependencies of `st`.
static sixbit_status add_switch_node(cudaStream_t st, cudaStream_t body_stream, cudaGraphConditionalHandle handle,
                                     int nbranches, sixbit_switch** out) {
  cudaStreamCaptureStatus status;
  cudaGraph_t graph = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edges = nullptr;
  size_t ndeps = 0;
  if (cudaStreamGetCaptureInfo(st, &status, nullptr, &graph, &deps, &edges, &ndeps) != cudaSuccess)
    return SIXBIT_ECUDA;
  if (status != cudaStreamCaptureStatusActive || graph == nullptr) return SIXBIT_EINVAL;
  cudaGraphNodeParams params = {};
  params.type = cudaGraphNodeTypeConditional;
  params.conditional.handle = handle;
  params.conditional.type = cudaGraphCondTypeSwitch;
  params.conditional.size = static_cast<unsigned int>(nbranches);
  cudaGraphNode_t node;
  if (cudaGraphAddNode(&node, graph, deps, edges, ndeps, &params) != cudaSuccess) return SIXBIT_ECUDA;
  if (cudaStreamUpdateCaptureDependencies(st, &node, nullptr, 1, cudaStreamSetCaptureDependencies) != cudaSuccess)
    return SIXBIT_ECUDA;

  sixbit_switch* sw = new (std::nothrow) sixbit_switch();
  if (sw == nullptr) return SIXBIT_EINVAL;
  sw->n = nbranches;
  sw->open_branch = -1;
  for (int i = 0; i < nbranches; ++i) sw->bodies[i] = params.conditional.phGraph_out[i];
  sw->body_stream = body_stream;
  *out = sw;
  return SIXBIT_OK;
}

extern "C" sixbit_status sixbit_graph_cond_create(void* stream, int nbranches, uint64_t* handle) {
  if (stream == nullptr || handle == nullptr || nbranches < 1 || nbranches > 8) return SIXBIT_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus status;
  cudaGraph_t graph = nullptr;
  if (cudaStreamGetCaptureInfo(st, &status, nullptr, &graph) != cudaSuccess) return SIXBIT_ECUDA;
  if (status != cudaStreamCaptureStatusActive || graph == nullptr) return SIXBIT_EINVAL;
  cudaGraphConditionalHandle h;
  if (cudaGraphConditionalHandleCreate(&h, graph, static_cast<unsigned int>(nbranches),
                                       cudaGraphCondAssignDefault) != cudaSuccess)
    return SIXBIT_ECUDA;
  *handle = static_cast<uint64_t>(h);
  return SIXBIT_OK;
}

extern "C" sixbit_status sixbit_graph_switch_begin_cond(void* stream, void* body_stream, uint64_t handle,
                                                        int nbranches, sixbit_switch** out) {
  if (stream == nullptr || body_stream == nullptr || body_stream == stream || out == nullptr || nbranches < 1 ||
      nbranches > 8)
    return SIXBIT_EINVAL;
  return add_switch_node(static_cast<cudaStream_t>(stream), static_cast<cudaStream_t>(body_stream),
                         static_cast<cudaGraphConditionalHandle>(handle), nbranches, out);
}

extern "C" sixbit_status sixbit_graph_branch_begin(sixbit_switch* sw, int branch, void** body_stream) {
  if (sw == nullptr || body_stream == nullptr || branch < 0 || branch >= sw->n || sw->open_branch >= 0)
    return SIXBIT_EINVAL;
  if (cudaStreamBeginCaptureToGraph(sw->body_stream, sw->bodies[branch], nullptr, nullptr, 0,
                                    cudaStreamCaptureModeRelaxed) != cudaSuccess)
    return SIXBIT_ECUDA;
  sw->open_branch = branch;
  *body_stream = sw->body_stream;
  return SIXBIT_OK;
}

extern "C" sixbit_status sixbit_graph_branch_end(sixbit_switch* sw) {
  if (sw == nullptr || sw->open_branch < 0) return SIXBIT_EINVAL;
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(sw->body_stream, &g);
  sw->open_branch = -1;
  return e == cudaSuccess ? SIXBIT_OK : SIXBIT_ECUDA;
}

extern "C" sixbit_status sixbit_graph_switch_end(sixbit_switch* sw) {
  if (sw == nullptr || sw->open_branch >= 0) return SIXBIT_EINVAL;
  delete sw;
  return SIXBIT_OK;
}
