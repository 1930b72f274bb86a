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
// Design (HBM-bound): the gate is one scalar per token, a reduction over the
// full hidden row; the conv is per channel along the token axis. The fused
// kernel takes a tile of TT consecutive tokens and
//   1. reduces the gate scalars of the tile and of its dilation halo (the
//      (K-1)*d previous tokens of the same request) with one warp per token
//      (16-byte loads, warp-shuffle reductions) into shared memory;
//   2. walks the channels in chunks of CH: stages u = bf16(g * v) for the
//      tile + halo in shared memory (the dilation window), then every thread
//      produces 8 channels of one token from the K staged taps;
//   3. writes the carry-over state of every request that ends in the tile.
// u never goes to global memory; h and k are read once (halo rows are
// re-read from L2 by the neighbouring tile), v once, y written once.
#include "common.cuh"

namespace ple {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 512;          // channels staged per pass
constexpr int kChunkVecs = kChunk / 8;
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

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
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
  sh = warp_sum(sh);
  sk = warp_sum(sk);
  sd = warp_sum(sd);
  const float inv_c = 1.0f / static_cast<float>(C);
  const float score = sd / (sqrtf(fmaf(sh, inv_c, eps)) * sqrtf(fmaf(sk, inv_c, eps))) /
                      sqrtf(static_cast<float>(C));
  return 1.0f / (1.0f + expf(-score));
}

// ---------------------------------------------------------------------------
// ple_gate: one warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
gate_kernel(const ple_bf16_t* __restrict__ hidden, const ple_bf16_t* __restrict__ kv,
            const ple_bf16_t* __restrict__ gamma_h, const ple_bf16_t* __restrict__ gamma_k,
            float eps, int64_t T, int C, ple_bf16_t* __restrict__ out,
            float* __restrict__ gate_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const ple_bf16_t* h_row = hidden + t * C;
  const ple_bf16_t* k_row = kv + t * 2 * C;
  const float g = gate_scalar(h_row, k_row, gamma_h, gamma_k, C, eps, lane);
  if (gate_out != nullptr && lane == 0) gate_out[t] = g;
  const ple_bf16_t* v_row = k_row + C;
#pragma unroll 4
  for (int c = lane * 8; c < C; c += 32 * 8) {
    float v[8];
    unpack8(ldg16(v_row + c), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= g;
    *reinterpret_cast<uint4*>(out + t * C + c) = pack8(v);
  }
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
  int TT;
};

template <bool GATED>
__global__ void __launch_bounds__(kThreads)
conv_kernel(const __grid_constant__ ConvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = (a.K - 1) * a.dil;
  const int rows = a.TT + W;
  const int C = a.C;
  const int64_t T = a.T;
  // shared layout: u_s [rows][kChunk] bf16 | w_s [K][kChunk] f32 | g_s [rows] f32
  //                | start_s, end_s [TT] i64 | req_s [TT] i32
  uint4* u_s = reinterpret_cast<uint4*>(smem);
  float* w_s = reinterpret_cast<float*>(smem + static_cast<size_t>(rows) * kChunk * 2);
  float* g_s = w_s + a.K * kChunk;
  int64_t* start_s = reinterpret_cast<int64_t*>(g_s + ((rows + 1) & ~1));
  int64_t* end_s = start_s + a.TT;
  int* req_s = reinterpret_cast<int*>(end_s + a.TT);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * a.TT;
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const int64_t src_off = GATED ? C : 0;  // v sits after k in kv

  if (blockIdx.x == 0)
    for (int i = tid; i < a.num_reqs + 1; i += kThreads)
      check_qsl(a.qsl, a.num_reqs, T, i, a.dev_err);

  for (int i = tid; i < a.TT; i += kThreads) {
    const int64_t t = t0 + i;
    int r = 0;
    int64_t s = 0, e = 0;
    if (t < T) {
      r = find_request(a.qsl, a.num_reqs, t);
      request_span(a.qsl, a.num_reqs, T, r, &s, &e);
    }
    req_s[i] = r;
    start_s[i] = s;
    end_s[i] = e;
  }
  __syncthreads();
  // Halo rows are needed only back to the start of the first tile token's
  // request; earlier rows belong to other requests.
  const int64_t lo = start_s[0];

  if constexpr (GATED) {
    for (int i = warp; i < rows; i += kWarps) {
      const int64_t j = t0 - W + i;
      float g = 0.f;
      if (j >= lo && j < T) {
        g = gate_scalar(a.hidden + j * C, a.src + j * src_pitch, a.gamma_h, a.gamma_k, C,
                        a.eps, lane);
        if (lane == 0 && a.gate_out != nullptr && i >= W) a.gate_out[j] = g;
      }
      if (lane == 0) g_s[i] = g;
    }
    __syncthreads();
  }

  for (int c0 = 0; c0 < C; c0 += kChunk) {
    for (int idx = tid; idx < a.K * kChunk; idx += kThreads) {
      const int i = idx / kChunk;
      const int c = c0 + idx % kChunk;
      w_s[idx] = (c < C) ? __bfloat162float(
                               reinterpret_cast<const __nv_bfloat16*>(a.w)[static_cast<int64_t>(c) * a.K + i])
                         : 0.f;
    }
    for (int idx = tid; idx < rows * kChunkVecs; idx += kThreads) {
      const int i = idx / kChunkVecs;
      const int cv = idx - i * kChunkVecs;
      const int64_t j = t0 - W + i;
      const int c = c0 + cv * 8;
      if (c < C && j >= lo && j < T) {
        uint4 v = ldg16(a.src + j * src_pitch + src_off + c);
        if constexpr (GATED) {
          float f[8];
          unpack8(v, f);
          const float g = g_s[i];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] *= g;
          v = pack8(f);
        }
        u_s[static_cast<size_t>(i) * kChunkVecs + cv] = v;
      }
    }
    __syncthreads();

    for (int idx = tid; idx < a.TT * kChunkVecs; idx += kThreads) {
      const int tt = idx / kChunkVecs;
      const int cv = idx - tt * kChunkVecs;
      const int64_t t = t0 + tt;
      const int c = c0 + cv * 8;
      if (t >= T || c >= C) continue;
      const int r = req_s[tt];
      const int64_t start = start_s[tt];
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int i = 0; i < a.K; ++i) {
        const int64_t j = t - static_cast<int64_t>(a.K - 1 - i) * a.dil;
        uint4 uv = make_uint4(0, 0, 0, 0);
        if (j >= start) {
          uv = u_s[static_cast<size_t>(j - t0 + W) * kChunkVecs + cv];
        } else if (a.state != nullptr) {
          const int64_t hp = W + (j - start);  // history row, oldest first
          if (hp >= 0) uv = ldg16(a.state + (static_cast<int64_t>(r) * W + hp) * C + c);
        }
        float u[8];
        unpack8(uv, u);
        const float* wi = w_s + i * kChunk + cv * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wi[e], u[e], acc[e]);
      }
      *reinterpret_cast<uint4*>(a.out + t * C + c) = pack8(acc);

      // Carry-over: the block holding a request's last token writes its state.
      if (a.state_out != nullptr && W > 0 && t == end_s[tt] - 1) {
        for (int jj = 0; jj < W; ++jj) {
          const int64_t srcj = t - W + 1 + jj;
          uint4 uv = make_uint4(0, 0, 0, 0);
          if (srcj >= start) {
            uv = u_s[static_cast<size_t>(srcj - t0 + W) * kChunkVecs + cv];
          } else if (a.state != nullptr && W + (srcj - start) >= 0) {
            uv = ldg16(a.state + (static_cast<int64_t>(r) * W + W + (srcj - start)) * C + c);
          }
          *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = uv;
        }
      }
    }
    __syncthreads();
  }

  // Requests with no tokens keep their state (block 0 copies it through).
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    const int vecs = C / 8;
    for (int r = 0; r < a.num_reqs; ++r) {
      int64_t s, e;
      request_span(a.qsl, a.num_reqs, T, r, &s, &e);
      if (e != s) continue;
      for (int idx = tid; idx < W * vecs; idx += kThreads) {
        const int64_t off = (static_cast<int64_t>(r) * W + idx / vecs) * C + (idx % vecs) * 8;
        const uint4 v = a.state ? ldg16(a.state + off) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(a.state_out + off) = v;
      }
    }
  }
}

size_t conv_smem_bytes(int TT, int K, int dil) {
  const int W = (K - 1) * dil;
  const int rows = TT + W;
  return static_cast<size_t>(rows) * kChunk * 2 + static_cast<size_t>(K) * kChunk * 4 +
         static_cast<size_t>((rows + 1) & ~1) * 4 + static_cast<size_t>(TT) * 16 +
         static_cast<size_t>(TT) * 4;
}

int pick_tile(int64_t T) {
  const int64_t target = 2 * static_cast<int64_t>(num_sms());
  int tt = 32;
  while (tt > 4 && (T + tt - 1) / tt < target) tt >>= 1;
  return tt;
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
  const int64_t blocks = (num_tokens + kWarps - 1) / kWarps;
  gate_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
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
  a.TT = pick_tile(T);
  const size_t smem = conv_smem_bytes(a.TT, K, dil);
  auto kernel = gated ? conv_kernel<true> : conv_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return check_cuda(err, name);
  const int64_t blocks = (T + a.TT - 1) / a.TT;
  if (blocks > 0x7fffffff) return fail(PLE_ERR_UNSUPPORTED, "%s: too many tokens", name);
  kernel<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(a);
  return check_cuda(cudaGetLastError(), name);
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
