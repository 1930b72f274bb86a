// Status text, device-property cache, event wait, version, tensor-map encoder.
#include "common.cuh"
#include "tma.cuh"

#include <cstdlib>

#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <thread>

namespace ple {

namespace {
thread_local char g_last_error[512] = "";
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
int g_smem[kMaxDevices] = {0};
}  // namespace

ple_status fail(ple_status status, const char* fmt, ...) {
  va_list args;
  va_start(args, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, args);
  va_end(args);
  return status;
}

ple_status check_cuda(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return PLE_OK;
  return fail(PLE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err),
              cudaGetErrorString(err));
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices && g_sms[dev] > 0) return g_sms[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices) g_sms[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int smem_per_sm() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && g_smem[dev] > 0) return g_smem[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (dev >= 0 && dev < kMaxDevices) g_smem[dev] = n;
  return n;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("PLE_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

ple_status copy_carry(void* dst, const void* src, size_t bytes,
                      cudaStream_t stream) {
  if (dst == nullptr || bytes == 0) return PLE_OK;
  cudaError_t err = (src != nullptr)
                        ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, stream)
                        : cudaMemsetAsync(dst, 0, bytes, stream);
  return check_cuda(err, "carry-over copy");
}

}  // namespace ple

PLE_EXPORT const char* ple_last_error(void) { return ple::g_last_error; }

PLE_EXPORT const char* ple_version(void) { return "libple 0.1 (sm_103a)"; }

PLE_EXPORT ple_status ple_wait(cudaEvent_t done, cudaStream_t consumer,
                               int32_t timeout_ms) {
  if (done == nullptr) return ple::fail(PLE_ERR_INVALID_ARG, "ple_wait: null event");
  if (timeout_ms > 0) {
    auto deadline = std::chrono::steady_clock::now() +
                    std::chrono::milliseconds(timeout_ms);
    for (;;) {
      cudaError_t q = cudaEventQuery(done);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) return ple::check_cuda(q, "ple_wait: cudaEventQuery");
      if (std::chrono::steady_clock::now() >= deadline)
        return ple::fail(PLE_ERR_TIMEOUT, "ple_wait: event not complete after %d ms",
                         timeout_ms);
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  return ple::check_cuda(cudaStreamWaitEvent(consumer, done, 0),
                         "ple_wait: cudaStreamWaitEvent");
}
