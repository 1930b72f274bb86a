// Step runtime of the end-to-end host path: CUDA graph capture of a layer's
// calls, and one step's enqueue across three streams (uploads on a copy-in
// stream, the layer on a compute stream, read-backs on a copy-out stream),
// ordered by events so that neighbouring steps overlap:
//   copy_in  waits `computed` (the slot's inputs may be overwritten once its
//            previous step has computed), uploads, records `loaded`;
//   compute  waits `loaded` and `returned` (the slot's output buffer may be
//            overwritten once its previous step has been read back), runs the
//            layer, records `computed`;
//   copy_out waits `computed`, reads back, records `returned`.
// An event that was never recorded is complete, so a slot's first step
// waits for nothing. Every copy is one cudaMemcpyAsync. Host code only.
#include "common.cuh"

#include <new>

struct ple_graph_s {
  cudaGraphExec_t exec;
};

namespace ple {
namespace {

ple_status check_copies(const ple_copy* copies, int32_t n, const char* name) {
  if (n < 0 || (n > 0 && copies == nullptr))
    return fail(PLE_ERR_INVALID_ARG, "%s: %d copies at %p", name, n,
                static_cast<const void*>(copies));
  for (int32_t i = 0; i < n; ++i)
    if (copies[i].bytes > 0 && (copies[i].dst == nullptr || copies[i].src == nullptr))
      return fail(PLE_ERR_INVALID_ARG, "%s: copy %d has a null pointer", name, i);
  return PLE_OK;
}

ple_status copy_all(const ple_copy* copies, int32_t n, cudaMemcpyKind kind, cudaStream_t stream,
                    const char* name) {
  for (int32_t i = 0; i < n; ++i) {
    if (copies[i].bytes == 0) continue;
    const cudaError_t err = cudaMemcpyAsync(copies[i].dst, copies[i].src, copies[i].bytes, kind,
                                            stream);
    if (err != cudaSuccess) return check_cuda(err, name);
  }
  return PLE_OK;
}

ple_status step_begin(cudaStream_t copy_in, cudaStream_t compute, const ple_copy* uploads,
                      int32_t num_uploads, cudaEvent_t loaded, cudaEvent_t computed,
                      cudaEvent_t returned, const char* name) {
  ple_status s = check_cuda(cudaStreamWaitEvent(copy_in, computed, 0), name);
  if (s != PLE_OK) return s;
  s = copy_all(uploads, num_uploads, cudaMemcpyHostToDevice, copy_in, name);
  if (s != PLE_OK) return s;
  s = check_cuda(cudaEventRecord(loaded, copy_in), name);
  if (s != PLE_OK) return s;
  s = check_cuda(cudaStreamWaitEvent(compute, loaded, 0), name);
  if (s != PLE_OK) return s;
  return check_cuda(cudaStreamWaitEvent(compute, returned, 0), name);
}

ple_status step_end(cudaStream_t compute, cudaStream_t copy_out, const ple_copy* downloads,
                    int32_t num_downloads, cudaEvent_t computed, cudaEvent_t returned,
                    const char* name) {
  ple_status s = check_cuda(cudaEventRecord(computed, compute), name);
  if (s != PLE_OK) return s;
  s = check_cuda(cudaStreamWaitEvent(copy_out, computed, 0), name);
  if (s != PLE_OK) return s;
  s = copy_all(downloads, num_downloads, cudaMemcpyDeviceToHost, copy_out, name);
  if (s != PLE_OK) return s;
  return check_cuda(cudaEventRecord(returned, copy_out), name);
}

bool streams_ok(cudaStream_t a, cudaStream_t b, cudaStream_t c) {
  return a != nullptr && b != nullptr && c != nullptr && a != b && b != c && a != c;
}

}  // namespace
}  // namespace ple

using namespace ple;

PLE_EXPORT ple_status ple_graph_begin(cudaStream_t stream) {
  if (stream == nullptr)
    return fail(PLE_ERR_INVALID_ARG, "ple_graph_begin: capture needs a created stream");
  return check_cuda(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal),
                    "ple_graph_begin");
}

PLE_EXPORT ple_status ple_graph_end(cudaStream_t stream, ple_graph* graph) {
  if (graph != nullptr) *graph = nullptr;
  if (stream == nullptr) return fail(PLE_ERR_INVALID_ARG, "ple_graph_end: null stream");
  cudaGraph_t g = nullptr;
  cudaError_t err = cudaStreamEndCapture(stream, &g);
  if (err != cudaSuccess) return check_cuda(err, "ple_graph_end: capture");
  if (graph == nullptr) {
    cudaGraphDestroy(g);
    return fail(PLE_ERR_INVALID_ARG, "ple_graph_end: null graph output (capture discarded)");
  }
  cudaGraphExec_t exec = nullptr;
  err = cudaGraphInstantiate(&exec, g, 0);
  cudaGraphDestroy(g);
  if (err != cudaSuccess) return check_cuda(err, "ple_graph_end: instantiate");
  ple_graph h = new (std::nothrow) ple_graph_s{exec};
  if (h == nullptr) {
    cudaGraphExecDestroy(exec);
    return fail(PLE_ERR_UNSUPPORTED, "ple_graph_end: out of host memory");
  }
  *graph = h;
  return PLE_OK;
}

PLE_EXPORT ple_status ple_graph_launch(ple_graph graph, cudaStream_t stream) {
  if (graph == nullptr) return fail(PLE_ERR_INVALID_ARG, "ple_graph_launch: null graph");
  return check_cuda(cudaGraphLaunch(graph->exec, stream), "ple_graph_launch");
}

PLE_EXPORT void ple_graph_destroy(ple_graph graph) {
  if (graph == nullptr) return;
  cudaGraphExecDestroy(graph->exec);
  delete graph;
}

PLE_EXPORT ple_status ple_event_create(cudaEvent_t* event) {
  if (event == nullptr) return fail(PLE_ERR_INVALID_ARG, "ple_event_create: null output");
  *event = nullptr;
  return check_cuda(cudaEventCreateWithFlags(event, cudaEventDisableTiming), "ple_event_create");
}

PLE_EXPORT void ple_event_destroy(cudaEvent_t event) {
  if (event != nullptr) cudaEventDestroy(event);
}

PLE_EXPORT ple_status ple_event_synchronize(cudaEvent_t event) {
  if (event == nullptr) return fail(PLE_ERR_INVALID_ARG, "ple_event_synchronize: null event");
  return check_cuda(cudaEventSynchronize(event), "ple_event_synchronize");
}

PLE_EXPORT ple_status ple_step_begin(cudaStream_t copy_in, cudaStream_t compute,
                                     const ple_copy* uploads, int32_t num_uploads,
                                     cudaEvent_t loaded, cudaEvent_t computed,
                                     cudaEvent_t returned) {
  const char* name = "ple_step_begin";
  if (copy_in == nullptr || compute == nullptr || copy_in == compute)
    return fail(PLE_ERR_INVALID_ARG, "%s: copy_in and compute must be two created streams", name);
  if (loaded == nullptr || computed == nullptr || returned == nullptr)
    return fail(PLE_ERR_INVALID_ARG, "%s: null event", name);
  const ple_status s = check_copies(uploads, num_uploads, name);
  if (s != PLE_OK) return s;
  return step_begin(copy_in, compute, uploads, num_uploads, loaded, computed, returned, name);
}

PLE_EXPORT ple_status ple_step_end(cudaStream_t compute, cudaStream_t copy_out,
                                   const ple_copy* downloads, int32_t num_downloads,
                                   cudaEvent_t computed, cudaEvent_t returned) {
  const char* name = "ple_step_end";
  if (compute == nullptr || copy_out == nullptr || compute == copy_out)
    return fail(PLE_ERR_INVALID_ARG, "%s: compute and copy_out must be two created streams", name);
  if (computed == nullptr || returned == nullptr)
    return fail(PLE_ERR_INVALID_ARG, "%s: null event", name);
  const ple_status s = check_copies(downloads, num_downloads, name);
  if (s != PLE_OK) return s;
  return step_end(compute, copy_out, downloads, num_downloads, computed, returned, name);
}

PLE_EXPORT ple_status ple_step(cudaStream_t copy_in, cudaStream_t compute, cudaStream_t copy_out,
                               const ple_copy* uploads, int32_t num_uploads, ple_graph graph,
                               const ple_copy* downloads, int32_t num_downloads,
                               cudaEvent_t loaded, cudaEvent_t computed, cudaEvent_t returned) {
  const char* name = "ple_step";
  if (!streams_ok(copy_in, compute, copy_out))
    return fail(PLE_ERR_INVALID_ARG, "%s: copy_in, compute and copy_out must be three created streams",
                name);
  if (graph == nullptr) return fail(PLE_ERR_INVALID_ARG, "%s: null graph", name);
  if (loaded == nullptr || computed == nullptr || returned == nullptr)
    return fail(PLE_ERR_INVALID_ARG, "%s: null event", name);
  ple_status s = check_copies(uploads, num_uploads, name);
  if (s == PLE_OK) s = check_copies(downloads, num_downloads, name);
  if (s != PLE_OK) return s;
  s = step_begin(copy_in, compute, uploads, num_uploads, loaded, computed, returned, name);
  if (s != PLE_OK) return s;
  s = check_cuda(cudaGraphLaunch(graph->exec, compute), name);
  if (s != PLE_OK) return s;
  return step_end(compute, copy_out, downloads, num_downloads, computed, returned, name);
}
