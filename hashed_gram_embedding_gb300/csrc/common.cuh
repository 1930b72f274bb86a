// Shared host/device helpers of libple (status text, device properties,
// small PTX wrappers). Every kernel of the library is in this directory.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ple.h"

#define PLE_EXPORT extern "C" __attribute__((visibility("default")))

namespace ple {

// Record a formatted reason for the status about to be returned; returns it.
ple_status fail(ple_status status, const char* fmt, ...);
// Map a CUDA error (from a launch or runtime call) to PLE_ERR_CUDA.
ple_status check_cuda(cudaError_t err, const char* what);
// Streaming multiprocessors of the current device (cached per device).
int num_sms();
// True if [a, a+na) and [b, b+nb) overlap (byte ranges).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  auto pa = reinterpret_cast<uintptr_t>(a);
  auto pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}
inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Copy a carry-over buffer (context / conv state) through when a call has
// no tokens, so ping-pong callers always find the next state in `dst`.
ple_status copy_carry(void* dst, const void* src, size_t bytes,
                      cudaStream_t stream);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void set_dev_err(int32_t* dev_err, int32_t bit) {
  if (dev_err != nullptr) atomicOr(dev_err, bit);
}

// Request of token t: last r with qsl[r] <= t, clamped to [0, R-1].
// Works (returns some r in range) whatever qsl holds.
__device__ __forceinline__ int find_request(const int32_t* __restrict__ qsl,
                                            int num_reqs, int64_t t) {
  int lo = 0, hi = num_reqs + 1;  // count of entries <= t lies in [lo, hi]
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(__ldg(qsl + mid)) <= t) lo = mid + 1; else hi = mid;
  }
  int r = lo - 1;
  r = r < 0 ? 0 : r;
  return r >= num_reqs ? num_reqs - 1 : r;
}

// Token span [start, end) of request r, clamped into [0, T] so that invalid
// contents of qsl can never produce an out-of-range access.
__device__ __forceinline__ void request_span(const int32_t* __restrict__ qsl,
                                             int num_reqs, int64_t T, int r,
                                             int64_t* start, int64_t* end) {
  int64_t s = __ldg(qsl + r);
  int64_t e = (r + 1 < num_reqs) ? static_cast<int64_t>(__ldg(qsl + r + 1)) : T;
  s = s < 0 ? 0 : (s > T ? T : s);
  e = e < s ? s : (e > T ? T : e);
  *start = s;
  *end = e;
}

// Block-level check of query_start_loc: qsl[0] == 0, non-decreasing,
// qsl[R] <= T. Any thread may call it for its share of r.
__device__ __forceinline__ void check_qsl(const int32_t* __restrict__ qsl,
                                          int num_reqs, int64_t T, int64_t i,
                                          int32_t* dev_err) {
  if (i < num_reqs) {
    if (__ldg(qsl + i) > __ldg(qsl + i + 1)) set_dev_err(dev_err, PLE_DEVERR_QSL);
  }
  if (i == 0) {
    if (__ldg(qsl) != 0 || static_cast<int64_t>(__ldg(qsl + num_reqs)) > T)
      set_dev_err(dev_err, PLE_DEVERR_QSL);
  }
}

}  // namespace ple
