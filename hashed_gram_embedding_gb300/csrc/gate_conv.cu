// ple_gate, ple_conv, ple_gate_conv: RMSNorm + sigmoid gate and the dilated
// causal depthwise short conv over ragged requests.
//
// Sources: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), 实现拆解 item 2
// (_ple_gate_kernel: "PLE gating and normalisation"; _ple_conv_kernel: dilated
// short convolution), item 4 (short-conv cached state for decode), item 5
// (prefill / decode / spec-decode PyTorch references). The pages give neither
// formula; the readings implemented here are
//   g_t = sigmoid(<rms(h_t)*gamma_h, rms(k_t)*gamma_k> / sqrt(C)),
//   rms(x) = x / sqrt(mean(x^2) + eps),  u_t = bf16_rn(g_t * v_t),
//   y_t[c] = sum_{i<K} w[c][i] * u_{t-(K-1-i)*d}[c]
// over each request's virtual sequence (conv state ++ segment, zeros before).
//
// Design (HBM-bound: read h, k, v once, write y once; u never leaves the SM).
// One 768-thread CTA per SM owns a contiguous token range [t0, t1):
//   1. gate: one warp per row reduces sum h^2, sum k^2 and sum h*k*gh*gk over
//      the full hidden row (16-byte loads, four 256-channel blocks of loads in
//      flight per lane, warp-shuffle reductions) for the range and its
//      dilation halo (the (K-1)*d previous tokens of the same request); the
//      gate scalars go to shared memory;
//   2. conv: a walker owns 8 channels and one residue class mod d of a
//      segment of the range; since the taps of y_t are t, t-d, ..., t-(K-1)d,
//      a ring of K gated values in registers holds the whole dilation window
//      whatever d is: u = bf16(g*v) is computed once per token and every tap
//      is a register read. Crossing into a new request reloads the ring from
//      that request's carry-over state (or zeros); the walker holding a
//      request's last token writes the new state.
#include "common.cuh"

#include <cstdlib>

namespace ple {
namespace {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kConvThreads = 768;
constexpr int kConvWarps = kConvThreads / 32;
constexpr int kMaxK = 8;
constexpr int kMaxHalo = 64;

__device__ __forceinline__ uint4 ldg16(const ple_bf16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void unpack8(uint4 v, float f[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(b[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
  uint4 v;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) b[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
  return v;
}

// u = bf16(g * v) for 8 packed bf16 values.
__device__ __forceinline__ uint4 gate8(uint4 v, float g) {
  float f[8];
  unpack8(v, f);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] *= g;
  return pack8(f);
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

// Gate scalar of one token, computed by a whole warp; every lane gets it.
__device__ __forceinline__ float gate_scalar(const ple_bf16_t* __restrict__ h_row,
                                             const ple_bf16_t* __restrict__ k_row,
                                             const ple_bf16_t* __restrict__ gamma_h,
                                             const ple_bf16_t* __restrict__ gamma_k,
                                             int C, float eps, int lane) {
  float sh = 0.f, sk = 0.f, sd = 0.f;
#pragma unroll 4
  for (int c = lane * 8; c < C; c += 32 * 8) {
    float h[8], k[8], gh[8], gk[8];
    unpack8(ldg16(h_row + c), h);
    unpack8(ldg16(k_row + c), k);
    unpack8(ldg16(gamma_h + c), gh);
    unpack8(ldg16(gamma_k + c), gk);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sh = fmaf(h[e], h[e], sh);
      sk = fmaf(k[e], k[e], sk);
      sd = fmaf(h[e] * gh[e], k[e] * gk[e], sd);
    }
  }
  return gate_of(warp_sum(sh), warp_sum(sk), warp_sum(sd), C, eps);
}

// ---------------------------------------------------------------------------
// ple_gate: one warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGateThreads)
gate_kernel(const ple_bf16_t* __restrict__ hidden, const ple_bf16_t* __restrict__ kv,
            const ple_bf16_t* __restrict__ gamma_h, const ple_bf16_t* __restrict__ gamma_k,
            float eps, int64_t T, int C, ple_bf16_t* __restrict__ out,
            float* __restrict__ gate_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kGateWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const ple_bf16_t* h_row = hidden + t * C;
  const ple_bf16_t* k_row = kv + t * 2 * C;
  const float g = gate_scalar(h_row, k_row, gamma_h, gamma_k, C, eps, lane);
  if (gate_out != nullptr && lane == 0) gate_out[t] = g;
  const ple_bf16_t* v_row = k_row + C;
#pragma unroll 4
  for (int c = lane * 8; c < C; c += 32 * 8)
    *reinterpret_cast<uint4*>(out + t * C + c) = gate8(ldg16(v_row + c), g);
}

// ---------------------------------------------------------------------------
// ple_conv (GATED = false, input x) and ple_gate_conv (GATED = true).
// ---------------------------------------------------------------------------
struct ConvArgs {
  const ple_bf16_t* hidden;   // gated only
  const ple_bf16_t* src;      // kv (gated) or x (plain)
  const ple_bf16_t* gamma_h;
  const ple_bf16_t* gamma_k;
  float eps;
  const int32_t* qsl;
  int num_reqs;
  int64_t T;
  int C;
  const ple_bf16_t* w;
  int K;
  int dil;
  const ple_bf16_t* state;
  ple_bf16_t* state_out;
  ple_bf16_t* out;
  float* gate_out;
  int32_t* dev_err;
};

// Walks one (8-channel group, residue class rho mod d, token segment) of the
// CTA's range: tokens t = s0 + rho, s0 + rho + d, ... < s1. The taps of y_t
// sit at t, t-d, ..., t-(K-1)d -- all in the walker's own residue class -- so
// a ring of K gated values (registers) holds the whole dilation window:
// ring[i] = u of token t - (K-1-i)*d, and y_t = sum_i w[i] * ring[i].
template <bool GATED, int KT>
struct ConvWalker {
  const ConvArgs& a;
  const float* g_s;      // gate scalars, row i <-> token row0 + i
  int64_t row0;          // t0 - W
  int W, dil, C, c;
  int64_t src_pitch, src_off;
  uint4 wt[KT];          // taps of this thread's 8 channels, packed bf16

  __device__ ConvWalker(const ConvArgs& args, const float* g, int64_t t0, int c_)
      : a(args), g_s(g), c(c_) {
    dil = a.dil;
    W = (KT - 1) * dil;
    C = a.C;
    row0 = t0 - W;
    src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
    src_off = GATED ? C : 0;
    const uint16_t* w = reinterpret_cast<const uint16_t*>(a.w);
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      uint32_t p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        p[e] = static_cast<uint32_t>(__ldg(w + static_cast<int64_t>(c + 2 * e) * KT + i)) |
               (static_cast<uint32_t>(__ldg(w + static_cast<int64_t>(c + 2 * e + 1) * KT + i)) << 16);
      wt[i] = make_uint4(p[0], p[1], p[2], p[3]);
    }
  }

  // gated (or plain) input of token j of request r whose first token is start
  __device__ __forceinline__ uint4 input(int64_t j, int r, int64_t start) const {
    if (j >= start) {
      const uint4 v = ldg16(a.src + j * src_pitch + src_off + c);
      if constexpr (GATED) return gate8(v, g_s[j - row0]);
      return v;
    }
    const int64_t hp = W + (j - start);  // history row, oldest first
    if (a.state != nullptr && hp >= 0)
      return ldg16(a.state + (static_cast<int64_t>(r) * W + hp) * C + c);
    return make_uint4(0, 0, 0, 0);
  }

  __device__ __forceinline__ static void fma8(float acc[8], uint4 w, uint4 u) {
    float f[8], g[8];
    unpack8(u, f);
    unpack8(w, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(g[e], f[e], acc[e]);
  }

  // Next request that owns token t (skips empty requests).
  __device__ __forceinline__ void advance(int64_t t, int* r, int64_t* start, int64_t* end) const {
    do {
      ++*r;
      request_span(a.qsl, a.num_reqs, a.T, *r, start, end);
    } while (*end <= t && *r + 1 < a.num_reqs);
  }

  __device__ void run(int64_t s0, int64_t s1, int rho) {
    int64_t t = s0 + rho;
    if (t >= s1) return;
    int r = find_request(a.qsl, a.num_reqs, t);
    int64_t start, end;
    request_span(a.qsl, a.num_reqs, a.T, r, &start, &end);
    uint4 ring[KT];
#pragma unroll
    for (int i = 0; i < KT - 1; ++i)
      ring[i + 1] = input(t - static_cast<int64_t>(KT - 1 - i) * dil, r, start);
    for (; t < s1; t += dil) {
      if (t >= end) {  // a new request: reload the window from its history
        advance(t, &r, &start, &end);
#pragma unroll
        for (int i = 0; i < KT - 1; ++i)
          ring[i + 1] = input(t - static_cast<int64_t>(KT - 1 - i) * dil, r, start);
      }
#pragma unroll
      for (int i = 0; i < KT - 1; ++i) ring[i] = ring[i + 1];
      ring[KT - 1] = input(t, r, start);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < KT; ++i) fma8(acc, wt[i], ring[i]);
      *reinterpret_cast<uint4*>(a.out + t * C + c) = pack8(acc);
      // The walker holding a request's last token writes its new state: the
      // last W inputs of the request's virtual sequence (any residue class).
      if (a.state_out != nullptr && W > 0 && t == end - 1) {
        for (int jj = 0; jj < W; ++jj) {
          const uint4 u = input(t - W + 1 + jj, r, start);
          *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = u;
        }
      }
    }
  }
};

template <bool GATED, int KT>
__global__ void __launch_bounds__(kConvThreads, 1)
conv_kernel(const __grid_constant__ ConvArgs a) {
  extern __shared__ float g_s[];
  const int dil = a.dil;
  const int W = (KT - 1) * dil;
  const int C = a.C;
  const int64_t T = a.T;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t t0 = T * blockIdx.x / gridDim.x;
  const int64_t t1 = T * (blockIdx.x + 1) / gridDim.x;

  if (blockIdx.x == 0)
    for (int i = tid; i < a.num_reqs + 1; i += kConvThreads)
      check_qsl(a.qsl, a.num_reqs, T, i, a.dev_err);

  // Rows before the start of t0's request belong to other requests.
  int64_t lo, lo_end;
  request_span(a.qsl, a.num_reqs, T, find_request(a.qsl, a.num_reqs, t0), &lo, &lo_end);
  const int64_t row0 = t0 - W;

  // 1. gate scalars of rows [max(lo, row0), t1), one warp per row
  if constexpr (GATED) {
    const int64_t first = lo > row0 ? lo : row0;
    for (int64_t j = first + warp; j < t1; j += kConvWarps) {
      const float g = gate_scalar(a.hidden + j * C, a.src + j * 2 * static_cast<int64_t>(C),
                                  a.gamma_h, a.gamma_k, C, a.eps, lane);
      if (lane == 0) {
        g_s[j - row0] = g;
        if (a.gate_out != nullptr && j >= t0) a.gate_out[j] = g;
      }
    }
    __syncthreads();
  }

  // 2. the conv: walkers (channel group, residue class, segment)
  const int ng = C / 8;
  const int64_t n = t1 - t0;
  const int64_t per_seg = static_cast<int64_t>(ng) * dil;
  int64_t segs = kConvThreads / per_seg;
  if (segs < 1) segs = 1;
  const int64_t max_segs = (n + dil - 1) / dil;
  if (segs > max_segs) segs = max_segs > 0 ? max_segs : 1;
  for (int64_t item = tid; item < per_seg * segs; item += kConvThreads) {
    const int cg = static_cast<int>(item % ng);
    const int rho = static_cast<int>((item / ng) % dil);
    const int64_t seg = item / per_seg;
    ConvWalker<GATED, KT> walker(a, g_s, t0, cg * 8);
    walker.run(t0 + n * seg / segs, t0 + n * (seg + 1) / segs, rho);
  }

  // Requests with no tokens keep their state (CTA 0 copies it through).
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    for (int r = 0; r < a.num_reqs; ++r) {
      int64_t s, e;
      request_span(a.qsl, a.num_reqs, T, r, &s, &e);
      if (e != s) continue;
      for (int idx = tid; idx < W * ng; idx += kConvThreads) {
        const int64_t off = (static_cast<int64_t>(r) * W + idx / ng) * C + (idx % ng) * 8;
        const uint4 v = a.state ? ldg16(a.state + off) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(a.state_out + off) = v;
      }
    }
  }
}

ple_status validate_conv(const int32_t* qsl, int32_t num_reqs, int64_t T, int32_t C,
                         const ple_bf16_t* w, int32_t K, int32_t dil,
                         const ple_bf16_t* state, ple_bf16_t* state_out, const char* name) {
  if (T < 0 || C < 8 || C % 8 != 0)
    return fail(PLE_ERR_INVALID_ARG, "%s: hidden_size %d must be a positive multiple of 8", name, C);
  if (K < 1 || K > kMaxK || dil < 1 || (K - 1) * dil > kMaxHalo)
    return fail(PLE_ERR_INVALID_ARG, "%s: kernel_size %d / dilation %d out of range", name, K, dil);
  if (num_reqs < 0 || (num_reqs == 0 && T > 0))
    return fail(PLE_ERR_INVALID_ARG, "%s: num_reqs must be >= 1 when there are tokens", name);
  if (!w || (T > 0 && !qsl)) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  const size_t state_bytes = static_cast<size_t>(num_reqs) * (K - 1) * dil * C * 2;
  if (state && state_out && state_bytes > 0 && overlaps(state, state_bytes, state_out, state_bytes))
    return fail(PLE_ERR_INVALID_ARG, "%s: conv_state_out overlaps conv_state", name);
  if ((state && !aligned16(state)) || (state_out && !aligned16(state_out)))
    return fail(PLE_ERR_INVALID_ARG, "%s: state buffers must be 16-byte aligned", name);
  return PLE_OK;
}

// CTAs of the conv grid: one per SM, fewer when there are under 16 tokens per
// SM. PLE_CONV_CTAS overrides the count (launch-shape sweeps).
int conv_grid(int64_t T) {
  int64_t g = num_sms();
  const int64_t by_tokens = (T + 15) / 16;
  if (by_tokens < g) g = by_tokens;
  if (const char* e = getenv("PLE_CONV_CTAS")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 65535) g = v;
  }
  if (g > T) g = T;
  return static_cast<int>(g < 1 ? 1 : g);
}

template <bool GATED>
ple_status launch_conv(const ConvArgs& a, cudaStream_t stream, const char* name) {
  const int grid = conv_grid(a.T);
  const int64_t rows_max = (a.T + grid - 1) / grid + 1 + static_cast<int64_t>(a.K - 1) * a.dil;
  const size_t smem = GATED ? static_cast<size_t>(rows_max) * sizeof(float) : 0;
  if (smem > 200 * 1024)
    return fail(PLE_ERR_UNSUPPORTED, "%s: %zu bytes of gate scalars per CTA", name, smem);
  void (*kernel)(ConvArgs) = nullptr;
  switch (a.K) {
    case 1: kernel = conv_kernel<GATED, 1>; break;
    case 2: kernel = conv_kernel<GATED, 2>; break;
    case 3: kernel = conv_kernel<GATED, 3>; break;
    case 4: kernel = conv_kernel<GATED, 4>; break;
    case 5: kernel = conv_kernel<GATED, 5>; break;
    case 6: kernel = conv_kernel<GATED, 6>; break;
    case 7: kernel = conv_kernel<GATED, 7>; break;
    default: kernel = conv_kernel<GATED, 8>; break;
  }
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return check_cuda(err, name);
  kernel<<<grid, kConvThreads, smem, stream>>>(a);
  return check_cuda(cudaGetLastError(), name);
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_gate(const ple_bf16_t* hidden, const ple_bf16_t* kv,
                               const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k,
                               float eps, int64_t num_tokens, int32_t hidden_size,
                               ple_bf16_t* out, float* gate_out, cudaStream_t stream) {
  using namespace ple;
  if (num_tokens < 0 || hidden_size < 8 || hidden_size % 8 != 0)
    return fail(PLE_ERR_INVALID_ARG, "ple_gate: hidden_size %d must be a positive multiple of 8",
                hidden_size);
  if (num_tokens == 0) return PLE_OK;
  if (!hidden || !kv || !gamma_h || !gamma_k || !out)
    return fail(PLE_ERR_INVALID_ARG, "ple_gate: null pointer");
  if (!aligned16(hidden) || !aligned16(kv) || !aligned16(gamma_h) || !aligned16(gamma_k) ||
      !aligned16(out))
    return fail(PLE_ERR_INVALID_ARG, "ple_gate: buffers must be 16-byte aligned");
  const int64_t blocks = (num_tokens + kGateWarps - 1) / kGateWarps;
  gate_kernel<<<static_cast<unsigned>(blocks), kGateThreads, 0, stream>>>(
      hidden, kv, gamma_h, gamma_k, eps, num_tokens, hidden_size, out, gate_out);
  return check_cuda(cudaGetLastError(), "ple_gate launch");
}

static ple_status conv_entry(bool gated, const ple_bf16_t* hidden, const ple_bf16_t* src,
                             const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k, float eps,
                             const int32_t* qsl, int32_t num_reqs, int64_t T, int32_t C,
                             const ple_bf16_t* w, int32_t K, int32_t dil,
                             const ple_bf16_t* state, ple_bf16_t* state_out, ple_bf16_t* out,
                             float* gate_out, int32_t* dev_err, cudaStream_t stream,
                             const char* name) {
  using namespace ple;
  ple_status s = validate_conv(qsl, num_reqs, T, C, w, K, dil, state, state_out, name);
  if (s != PLE_OK) return s;
  const size_t state_bytes = static_cast<size_t>(num_reqs) * (K - 1) * dil * C * 2;
  if (T == 0) return copy_carry(state_out, state, state_bytes, stream);
  if (!src || !out || (gated && (!hidden || !gamma_h || !gamma_k)))
    return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(src) || !aligned16(out) ||
      (gated && (!aligned16(hidden) || !aligned16(gamma_h) || !aligned16(gamma_k))))
    return fail(PLE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", name);
  ConvArgs a{};
  a.hidden = hidden;
  a.src = src;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.eps = eps;
  a.qsl = qsl;
  a.num_reqs = num_reqs;
  a.T = T;
  a.C = C;
  a.w = w;
  a.K = K;
  a.dil = dil;
  a.state = state;
  a.state_out = state_out;
  a.out = out;
  a.gate_out = gate_out;
  a.dev_err = dev_err;
  return gated ? launch_conv<true>(a, stream, name) : launch_conv<false>(a, stream, name);
}

PLE_EXPORT ple_status ple_conv(const ple_bf16_t* x, const int32_t* query_start_loc,
                               int32_t num_reqs, int64_t num_tokens, int32_t hidden_size,
                               const ple_bf16_t* w, int32_t kernel_size, int32_t dilation,
                               const ple_bf16_t* conv_state, ple_bf16_t* conv_state_out,
                               ple_bf16_t* out, int32_t* dev_err, cudaStream_t stream) {
  return conv_entry(false, nullptr, x, nullptr, nullptr, 0.f, query_start_loc, num_reqs,
                    num_tokens, hidden_size, w, kernel_size, dilation, conv_state,
                    conv_state_out, out, nullptr, dev_err, stream, "ple_conv");
}

PLE_EXPORT ple_status ple_gate_conv(const ple_bf16_t* hidden, const ple_bf16_t* kv,
                                    const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k,
                                    float eps, const int32_t* query_start_loc,
                                    int32_t num_reqs, int64_t num_tokens,
                                    int32_t hidden_size, const ple_bf16_t* w,
                                    int32_t kernel_size, int32_t dilation,
                                    const ple_bf16_t* conv_state,
                                    ple_bf16_t* conv_state_out, ple_bf16_t* out,
                                    float* gate_out, int32_t* dev_err,
                                    cudaStream_t stream) {
  return conv_entry(true, hidden, kv, gamma_h, gamma_k, eps, query_start_loc, num_reqs,
                    num_tokens, hidden_size, w, kernel_size, dilation, conv_state,
                    conv_state_out, out, gate_out, dev_err, stream, "ple_gate_conv");
}
