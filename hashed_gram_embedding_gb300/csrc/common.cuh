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
// Shared memory per SM of the current device, bytes (cached per device).
int smem_per_sm();
// True if [a, a+na) and [b, b+nb) overlap (byte ranges).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  auto pa = reinterpret_cast<uintptr_t>(a);
  auto pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}
inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Programmatic dependent launch. Every libple kernel is launched with
// programmatic stream serialization, so it may begin while the kernel before
// it in the stream is finishing: it first does set-up that touches no global
// memory (barriers, tensor memory, tensor-map prefetch), then pdl_wait()
// (griddepcontrol.wait: the previous grid has completed and its writes are
// visible) before its first global load or store, then pdl_trigger()
// (griddepcontrol.launch_dependents) so the next kernel may start launching.
// PLE_PDL=0 launches without the attribute (both instructions are then
// no-ops).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t stream, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl && pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, unsigned cluster, Args&&... args) {
  return launch_kernel_pdl(true, kernel, grid, block, smem, stream, cluster,
                           static_cast<Args&&>(args)...);
}

// Copy a carry-over buffer (context / conv state) through when a call has
// no tokens, so ping-pong callers always find the next state in `dst`.
ple_status copy_carry(void* dst, const void* src, size_t bytes,
                      cudaStream_t stream);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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

// ---------------------------------------------------------------------------
// mbarrier helpers (shared by the TMA-fed kernels). Every wait is bounded.
// ---------------------------------------------------------------------------

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s of %globaltimer per wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up after
// kWaitLimitNs, or early when `abort_flag` is set (if non-null).
__device__ __noinline__ inline bool mbar_wait(uint32_t bar, uint32_t parity,
                                              const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk async copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// bf16 / packed-float helpers and the gate scalar (ple_gate, ple_gate_conv
// and the fused reduction of ple_kv_proj_gate compute g with the same code)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ldg16(const ple_bf16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// bf16 pair word -> its two float32 values (low half is the first element).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(uint4 v, float f[8]) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
  f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
  f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Packed float32 pairs (sm_100+ two-wide FMA/MUL; each lane is an IEEE
// single-precision operation, identical to fmaf / __fmul_rn on that lane).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// lo += w.lo * x.lo, hi += w.hi * x.hi for two bf16 pair words, float32
// accumulators (sm_100+ mixed-precision FMA: the bf16 operands are exact in
// float32 and the product-sum is rounded once, so each lane equals fmaf on
// the unpacked values).
__device__ __forceinline__ void bf2_fma(uint32_t w, uint32_t x, float& lo, float& hi) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(lo), "+f"(hi) : "r"(w), "r"(x));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float gate_of(float sh, float sk, float sd, int C, float eps) {
  const float inv_c = 1.0f / static_cast<float>(C);
  const float score = sd / (sqrtf(fmaf(sh, inv_c, eps)) * sqrtf(fmaf(sk, inv_c, eps))) /
                      sqrtf(static_cast<float>(C));
  return 1.0f / (1.0f + expf(-score));
}

}  // namespace ple
