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
// Design (HBM-bound: read h, k, v once, write y once; u never reaches HBM):
//   pass 1 (gate_scalar_kernel): one warp per token reduces sum h^2, sum k^2
//     and sum h*k*gh*gk over the hidden row (16-byte loads, four blocks of
//     loads in flight per lane, warp-shuffle reductions) and writes the gate
//     scalar g_t (4 bytes per token) -- many warps per SM keep enough loads in
//     flight to stream h and k near the HBM rate;
//   pass 2 (conv_kernel<GATED=true>): a CTA takes a tile of tokens and a
//     256-channel slice, stages its dilation window -- the gated values
//     u = bf16(g*v) of the tile and of the (K-1)*d tokens before it, inside
//     the same request -- in shared memory with coalesced 16-byte loads, then
//     each lane owns 8 channels (taps in registers) and each warp walks tokens:
//     y_t = sum_i w_i * u_{t-(K-1-i)d} from shared memory (or from the
//     carry-over state before a request's first token). The CTA holding a
//     request's last token writes the request's new state for its channels.
// ple_conv is pass 2 on an ungated input; ple_gate is pass 1 plus u = g*v.
#include "common.cuh"

#include <cstdlib>

namespace ple {
namespace {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kConvThreads = 256;
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

// gamma_h[c] * gamma_k[c] for 8 channels, from the two bf16 vectors.
struct GammaFromGlobal {
  const ple_bf16_t* gh;
  const ple_bf16_t* gk;
  __device__ __forceinline__ void operator()(int c, float out[8]) const {
    float a[8], b[8];
    unpack8(ldg16(gh + c), a);
    unpack8(ldg16(gk + c), b);
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = a[e] * b[e];
  }
};

// Gate scalar of one token, computed by a whole warp; every lane gets it.
// <rms(h)*gh, rms(k)*gk> = sum(h*k*gh*gk) / (rms_h * rms_k).
template <class Gamma>
__device__ __forceinline__ float gate_scalar(const ple_bf16_t* __restrict__ h_row,
                                             const ple_bf16_t* __restrict__ k_row,
                                             const Gamma& gamma, int C, float eps, int lane) {
  float sh = 0.f, sk = 0.f, sd = 0.f;
#pragma unroll 4
  for (int c = lane * 8; c < C; c += 32 * 8) {
    float h[8], k[8], g[8];
    unpack8(ldg16(h_row + c), h);
    unpack8(ldg16(k_row + c), k);
    gamma(c, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sh = fmaf(h[e], h[e], sh);
      sk = fmaf(k[e], k[e], sk);
      sd = fmaf(h[e] * k[e], g[e], sd);
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
  const float g = gate_scalar(h_row, k_row, GammaFromGlobal{gamma_h, gamma_k}, C, eps, lane);
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

// gamma_h[c] * gamma_k[c], precomputed once per CTA in shared memory (the
// same float32 products GammaFromGlobal forms, so both kernels agree bit for
// bit).
struct GammaFromShared {
  const float* gg;
  __device__ __forceinline__ void operator()(int c, float out[8]) const {
    const float4 x = *reinterpret_cast<const float4*>(gg + c);
    const float4 y = *reinterpret_cast<const float4*>(gg + c + 4);
    out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
    out[4] = y.x; out[5] = y.y; out[6] = y.z; out[7] = y.w;
  }
};

constexpr int kGateScalarThreads = 512;
constexpr int kGateScalarWarps = kGateScalarThreads / 32;

// Pass 1 of ple_gate_conv: the gate scalars only, one warp per token.
__global__ void __launch_bounds__(kGateScalarThreads)
gate_scalar_kernel(const ple_bf16_t* __restrict__ hidden, const ple_bf16_t* __restrict__ kv,
                   const ple_bf16_t* __restrict__ gamma_h, const ple_bf16_t* __restrict__ gamma_k,
                   float eps, int64_t T, int C, float* __restrict__ gate_out) {
  extern __shared__ __align__(16) float gg_s[];  // [C]
  for (int c = threadIdx.x * 8; c < C; c += kGateScalarThreads * 8) {
    float f[8];
    GammaFromGlobal{gamma_h, gamma_k}(c, f);
    *reinterpret_cast<float4*>(gg_s + c) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(gg_s + c + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kGateScalarWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float g = gate_scalar(hidden + t * C, kv + t * 2 * C, GammaFromShared{gg_s}, C, eps, lane);
  if (lane == 0) gate_out[t] = g;
}

constexpr int kConvSlice = 256;            // channels per CTA (8 per lane)
constexpr int kConvSliceVecs = kConvSlice / 8;

// Pass 2: the dilated causal depthwise conv of one (token tile, channel
// slice); GATED: its input is u = bf16(g * v) with g from pass 1.
template <bool GATED, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_kernel(const __grid_constant__ ConvArgs a, const float* __restrict__ g, int tile_tokens) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int dil = a.dil;
  const int W = (K - 1) * dil;
  const int C = a.C;
  const int64_t T = a.T;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tile_tokens;
  const int64_t t1 = t0 + tile_tokens < T ? t0 + tile_tokens : T;
  const int n_tok = static_cast<int>(t1 - t0);
  const int c0 = blockIdx.y * kConvSlice;
  const int64_t row0 = t0 - W;                 // window row i <-> token row0 + i
  const int rows = n_tok + W;
  uint4* win = reinterpret_cast<uint4*>(smem);  // [rows][kConvSliceVecs]
  int4* tok_s = reinterpret_cast<int4*>(smem + static_cast<size_t>(tile_tokens + W) * kConvSlice * 2);
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const int64_t src_off = GATED ? C : 0;       // v sits after k in kv

  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = tid; i < a.num_reqs + 1; i += kConvThreads)
      check_qsl(a.qsl, a.num_reqs, T, i, a.dev_err);

  // request (start, end, index) of every tile token
  for (int i = tid; i < n_tok; i += kConvThreads) {
    const int r = find_request(a.qsl, a.num_reqs, t0 + i);
    int64_t st, en;
    request_span(a.qsl, a.num_reqs, T, r, &st, &en);
    tok_s[i] = make_int4(static_cast<int>(st - t0), static_cast<int>(en - t0), r, 0);
  }
  // window rows from the start of t0's request on (earlier rows belong to
  // other requests and are never read)
  int64_t lo, lo_end;
  request_span(a.qsl, a.num_reqs, T, find_request(a.qsl, a.num_reqs, t0), &lo, &lo_end);
  const int i_lo = static_cast<int>(lo > row0 ? lo - row0 : 0);
  // lanes past the last channel (C not a multiple of the slice) stay idle
  const bool active = c0 + lane * 8 < C;
  // one warp per window row: 32 lanes x 16 bytes = the slice's 512 bytes
  if (active) {
#pragma unroll 4
    for (int i = i_lo + warp; i < rows; i += kConvThreads / 32) {
      const int64_t j = row0 + i;
      uint4 v = ldg16(a.src + j * src_pitch + src_off + c0 + lane * 8);
      if constexpr (GATED) v = gate8(v, __ldg(g + j));
      win[i * kConvSliceVecs + lane] = v;
    }
  }
  __syncthreads();
  if (!active) return;

  // taps of this lane's 8 channels: w[c..c+7][0..K-1] is 8*K contiguous bf16
  // (K 16-byte loads), transposed into wt[tap][channel]
  float wt[K][8];
  {
    const uint4* wv = reinterpret_cast<const uint4*>(a.w + static_cast<int64_t>(c0 + lane * 8) * K);
#pragma unroll
    for (int q = 0; q < K; ++q) {
      float f[8];
      unpack8(__ldg(wv + q), f);  // elements 8q .. 8q+7 of the [8][K] block
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int flat = 8 * q + e;
        wt[flat % K][flat / K] = f[e];
      }
    }
  }
  const int c = c0 + lane * 8;
  for (int tt = warp; tt < n_tok; tt += kConvThreads / 32) {
    const int4 sr = tok_s[tt];
    const int64_t t = t0 + tt;
    const int64_t start = t0 + sr.x;
    const int r = sr.z;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const int64_t j = t - static_cast<int64_t>(K - 1 - i) * dil;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (j >= start) {
        u = win[static_cast<int>(j - row0) * kConvSliceVecs + lane];
      } else if (a.state != nullptr) {
        const int64_t hp = W + (j - start);  // history row, oldest first
        if (hp >= 0) u = ldg16(a.state + (static_cast<int64_t>(r) * W + hp) * C + c);
      }
      float f[8];
      unpack8(u, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(wt[i][e], f[e], acc[e]);
    }
    *reinterpret_cast<uint4*>(a.out + t * C + c) = pack8(acc);
    // carry-over: the CTA holding a request's last token writes its state
    if (a.state_out != nullptr && W > 0 && tt == sr.y - 1) {
      for (int jj = 0; jj < W; ++jj) {
        const int64_t sj = t - W + 1 + jj;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (sj >= start) u = win[static_cast<int>(sj - row0) * kConvSliceVecs + lane];
        else if (a.state != nullptr && W + (sj - start) >= 0)
          u = ldg16(a.state + (static_cast<int64_t>(r) * W + W + (sj - start)) * C + c);
        *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = u;
      }
    }
  }

  // Requests with no tokens keep their state (the first token tile copies it;
  // only active lanes get here).
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    for (int r = 0; r < a.num_reqs; ++r) {
      int64_t s0, e0;
      request_span(a.qsl, a.num_reqs, T, r, &s0, &e0);
      if (e0 != s0) continue;
      for (int jj = warp; jj < W; jj += kConvThreads / 32) {
        const int64_t off = (static_cast<int64_t>(r) * W + jj) * C + c;
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
  if (!aligned16(w)) return fail(PLE_ERR_INVALID_ARG, "%s: conv taps must be 16-byte aligned", name);
  const size_t state_bytes = static_cast<size_t>(num_reqs) * (K - 1) * dil * C * 2;
  if (state && state_out && state_bytes > 0 && overlaps(state, state_bytes, state_out, state_bytes))
    return fail(PLE_ERR_INVALID_ARG, "%s: conv_state_out overlaps conv_state", name);
  if ((state && !aligned16(state)) || (state_out && !aligned16(state_out)))
    return fail(PLE_ERR_INVALID_ARG, "%s: state buffers must be 16-byte aligned", name);
  return PLE_OK;
}

// Tokens per conv tile: 64 (halo overhead (K-1)d/64) unless that leaves
// fewer than ~4 CTAs per SM. PLE_CONV_TILE overrides (launch-shape sweeps).
int conv_tile_tokens(int64_t T, int C) {
  const int64_t slices = (C + kConvSlice - 1) / kConvSlice;
  int tile = 64;
  while (tile > 8 && ((T + tile - 1) / tile) * slices < 4 * static_cast<int64_t>(num_sms())) tile >>= 1;
  if (const char* e = getenv("PLE_CONV_TILE")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 256) tile = v;
  }
  return tile;
}

template <bool GATED>
ple_status launch_conv(const ConvArgs& a, const float* g, cudaStream_t stream, const char* name) {
  const int W = (a.K - 1) * a.dil;
  const int tile = conv_tile_tokens(a.T, a.C);
  const size_t smem = static_cast<size_t>(tile + W) * kConvSlice * 2 + static_cast<size_t>(tile) * 16;
  void (*kernel)(ConvArgs, const float*, int) = nullptr;
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
  const int64_t tiles = (a.T + tile - 1) / tile;
  if (tiles > 0x7fffffff) return fail(PLE_ERR_UNSUPPORTED, "%s: too many tokens", name);
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>((a.C + kConvSlice - 1) / kConvSlice));
  kernel<<<grid, kConvThreads, smem, stream>>>(a, g, tile);
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
  if (gated && gate_out == nullptr)
    return fail(PLE_ERR_INVALID_ARG, "%s: gate_out is required (it carries the gate scalars "
                "from the reduction pass to the conv pass)", name);
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
  if (!gated) return launch_conv<false>(a, nullptr, stream, name);
  const int64_t blocks = (T + kGateScalarWarps - 1) / kGateScalarWarps;
  const size_t gg_bytes = static_cast<size_t>(C) * sizeof(float);
  if (gg_bytes > 200 * 1024) return fail(PLE_ERR_UNSUPPORTED, "%s: hidden_size %d too large", name, C);
  cudaError_t ferr = cudaFuncSetAttribute(gate_scalar_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(gg_bytes));
  if (ferr != cudaSuccess) return check_cuda(ferr, name);
  gate_scalar_kernel<<<static_cast<unsigned>(blocks), kGateScalarThreads, gg_bytes, stream>>>(
      hidden, src, gamma_h, gamma_k, eps, T, C, gate_out);
  ple_status st = check_cuda(cudaGetLastError(), name);
  if (st != PLE_OK) return st;
  return launch_conv<true>(a, gate_out, stream, name);
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
