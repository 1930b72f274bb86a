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

#include <cooperative_groups.h>
#include <cstdlib>

namespace ple {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
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
//
// Grid: one thread-block cluster of CL CTAs per tile of TT tokens; CTA
// `part` of the cluster owns channels [part*slice, (part+1)*slice).
//   0. the tile's request boundaries (binary search) go to shared memory;
//   1. one thread issues bulk async copies of the v rows of the tile and its
//      halo (only rows of the first tile token's request or later) into
//      shared memory -- they land while step 2 runs;
//   2. (gated) warps reduce sum h^2, sum k^2, sum h*gh*k*gk over the CTA's
//      channel slice for every row; a cluster barrier publishes these partial
//      sums and every CTA adds the CL partials of each row through
//      distributed shared memory to get the gate scalars;
//   3. after the copies land, each thread produces 8 channels of one token:
//      u = bf16(g * v) for the K dilated taps (from shared memory, or the
//      carry-over state before the request's first token), fp32 FMA with
//      the taps, bf16 out; the CTA holding a request's last token writes that
//      request's new state for its channels.
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
  int TT;      // tokens per tile
  int CL;      // CTAs per tile (channel split; the cluster size when gated)
  int slice;   // channels per CTA (multiple of 8)
};

struct ConvSmem {
  // offsets in bytes from the dynamic shared-memory base
  size_t v, w, part, g, start, end, req, bar, total;
};

__host__ __device__ inline ConvSmem conv_smem_layout(int TT, int K, int dil, int slice) {
  ConvSmem L;
  const int rows = TT + (K - 1) * dil;
  size_t off = 0;
  L.v = off;      off += static_cast<size_t>(rows) * slice * 2;          // staged v rows
  off = (off + 15) & ~size_t(15);
  L.w = off;      off += static_cast<size_t>(K) * slice * 4;             // taps, [K][slice] f32
  L.part = off;   off += static_cast<size_t>(rows) * 4 * 4;              // partial sums
  L.g = off;      off += static_cast<size_t>(rows) * 4;                  // gate scalars
  off = (off + 7) & ~size_t(7);
  L.start = off;  off += static_cast<size_t>(TT) * 8;
  L.end = off;    off += static_cast<size_t>(TT) * 8;
  L.req = off;    off += static_cast<size_t>(TT) * 4;
  off = (off + 7) & ~size_t(7);
  L.bar = off;    off += 8;
  L.total = off;
  return L;
}

template <bool GATED>
__global__ void __launch_bounds__(kThreads)
conv_kernel(const __grid_constant__ ConvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int W = (a.K - 1) * a.dil;
  const int rows = a.TT + W;
  const int C = a.C;
  const int64_t T = a.T;
  const int slice = a.slice;
  const int ng = slice / 8;                      // 16-byte channel groups per CTA
  const ConvSmem L = conv_smem_layout(a.TT, a.K, a.dil, slice);
  uint4* v_s = reinterpret_cast<uint4*>(smem + L.v);
  float* w_s = reinterpret_cast<float*>(smem + L.w);
  float4* part_s = reinterpret_cast<float4*>(smem + L.part);
  float* g_s = reinterpret_cast<float*>(smem + L.g);
  int64_t* start_s = reinterpret_cast<int64_t*>(smem + L.start);
  int64_t* end_s = reinterpret_cast<int64_t*>(smem + L.end);
  int* req_s = reinterpret_cast<int*>(smem + L.req);
  const uint32_t bar = smem_u32(smem + L.bar);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int tile = blockIdx.x / a.CL;
  const int part = blockIdx.x % a.CL;
  const int c0 = part * slice;
  const int64_t t0 = static_cast<int64_t>(tile) * a.TT;
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const int64_t src_off = GATED ? C : 0;  // v sits after k in kv

  if (blockIdx.x == 0)
    for (int i = tid; i < a.num_reqs + 1; i += kThreads)
      check_qsl(a.qsl, a.num_reqs, T, i, a.dev_err);

  // 0. request of every tile token; taps of this CTA's channels
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
  for (int idx = tid; idx < a.K * slice; idx += kThreads) {
    const int i = idx / slice;
    const int c = c0 + idx - i * slice;
    w_s[idx] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.w)[static_cast<int64_t>(c) * a.K + i]);
  }
  for (int i = tid; i < rows; i += kThreads) part_s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // Halo rows are needed only back to the start of the first tile token's
  // request; earlier rows belong to other requests.
  const int64_t lo = start_s[0];
  const int i_lo = static_cast<int>(max(static_cast<int64_t>(0), lo - (t0 - W)));
  const int i_hi = static_cast<int>(min(static_cast<int64_t>(rows), T - (t0 - W)));

  // 1. stage v rows [i_lo, i_hi) of this CTA's channels
  if (tid == 0) {
    const uint32_t row_bytes = static_cast<uint32_t>(slice) * 2;
    const int n = i_hi > i_lo ? i_hi - i_lo : 0;
    mbar_arrive_expect_tx(bar, row_bytes * static_cast<uint32_t>(n));
    for (int i = i_lo; i < i_hi; ++i) {
      const int64_t j = t0 - W + i;
      bulk_copy_g2s(smem_u32(v_s) + static_cast<uint32_t>(i) * row_bytes,
                    a.src + j * src_pitch + src_off + c0, row_bytes, bar);
    }
  }

  // 2. gate scalars
  if constexpr (GATED) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int per_lane = (ng + 31) / 32;
    for (int i = i_lo + warp; i < i_hi; i += kWarps) {
      const int64_t j = t0 - W + i;
      const ple_bf16_t* h_row = a.hidden + j * C + c0;
      const ple_bf16_t* k_row = a.src + j * src_pitch + c0;
      float sh = 0.f, sk = 0.f, sd = 0.f;
      for (int m = 0; m < per_lane; ++m) {
        const int cv = lane + 32 * m;
        if (cv < ng) {
          float h[8], k[8], gh[8], gk[8];
          unpack8(ldg16(h_row + cv * 8), h);
          unpack8(ldg16(k_row + cv * 8), k);
          unpack8(ldg16(a.gamma_h + c0 + cv * 8), gh);
          unpack8(ldg16(a.gamma_k + c0 + cv * 8), gk);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            sh = fmaf(h[e], h[e], sh);
            sk = fmaf(k[e], k[e], sk);
            sd = fmaf(h[e] * gh[e], k[e] * gk[e], sd);
          }
        }
      }
      sh = warp_sum(sh);
      sk = warp_sum(sk);
      sd = warp_sum(sd);
      if (lane == 0) part_s[i] = make_float4(sh, sk, sd, 0.f);
    }
    cluster.sync();  // every CTA's partial sums are now visible cluster-wide
    const float inv_c = 1.0f / static_cast<float>(C);
    const float inv_sqrt_c = 1.0f / sqrtf(static_cast<float>(C));
    for (int i = i_lo + tid; i < i_hi; i += kThreads) {
      float sh = 0.f, sk = 0.f, sd = 0.f;
      for (int r = 0; r < a.CL; ++r) {
        const float4 p = *cluster.map_shared_rank(part_s + i, r);
        sh += p.x;
        sk += p.y;
        sd += p.z;
      }
      const float score = sd / (sqrtf(fmaf(sh, inv_c, a.eps)) * sqrtf(fmaf(sk, inv_c, a.eps))) *
                          inv_sqrt_c;
      const float g = 1.0f / (1.0f + expf(-score));
      g_s[i] = g;
      const int64_t j = t0 - W + i;
      if (part == 0 && a.gate_out != nullptr && i >= W) a.gate_out[j] = g;
    }
  }

  // 3. wait for the staged rows (bounded), then the dilated taps
  const bool staged = mbar_wait(bar, 0, nullptr);
  if (!staged && tid == 0) set_dev_err(a.dev_err, PLE_DEVERR_TIMEOUT);
  __syncthreads();

  if (staged) {
    for (int idx = tid; idx < a.TT * ng; idx += kThreads) {
      const int tt = idx / ng;
      const int cv = idx - tt * ng;
      const int64_t t = t0 + tt;
      if (t >= T) continue;
      const int c = c0 + cv * 8;
      const int r = req_s[tt];
      const int64_t start = start_s[tt];
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int i = 0; i < a.K; ++i) {
        const int64_t j = t - static_cast<int64_t>(a.K - 1 - i) * a.dil;
        float u[8];
        if (j >= start) {
          const int row = static_cast<int>(j - t0 + W);
          unpack8(v_s[static_cast<size_t>(row) * ng + cv], u);
          if constexpr (GATED) {
            const float g = g_s[row];
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = g * u[e];
            unpack8(pack8(u), u);  // u is rounded to bf16 before the conv
          }
        } else {
          const int64_t hp = W + (j - start);  // history row, oldest first
          uint4 hv = make_uint4(0, 0, 0, 0);
          if (a.state != nullptr && hp >= 0)
            hv = ldg16(a.state + (static_cast<int64_t>(r) * W + hp) * C + c);
          unpack8(hv, u);
        }
        const float4 w0 = *reinterpret_cast<const float4*>(w_s + i * slice + cv * 8);
        const float4 w1 = *reinterpret_cast<const float4*>(w_s + i * slice + cv * 8 + 4);
        acc[0] = fmaf(w0.x, u[0], acc[0]);
        acc[1] = fmaf(w0.y, u[1], acc[1]);
        acc[2] = fmaf(w0.z, u[2], acc[2]);
        acc[3] = fmaf(w0.w, u[3], acc[3]);
        acc[4] = fmaf(w1.x, u[4], acc[4]);
        acc[5] = fmaf(w1.y, u[5], acc[5]);
        acc[6] = fmaf(w1.z, u[6], acc[6]);
        acc[7] = fmaf(w1.w, u[7], acc[7]);
      }
      *reinterpret_cast<uint4*>(a.out + t * C + c) = pack8(acc);

      // Carry-over: the CTA holding a request's last token writes its state.
      if (a.state_out != nullptr && W > 0 && t == end_s[tt] - 1) {
        for (int jj = 0; jj < W; ++jj) {
          const int64_t sj = t - W + 1 + jj;
          uint4 sv = make_uint4(0, 0, 0, 0);
          if (sj >= start) {
            const int row = static_cast<int>(sj - t0 + W);
            sv = v_s[static_cast<size_t>(row) * ng + cv];
            if constexpr (GATED) {
              float u[8];
              unpack8(sv, u);
              const float g = g_s[row];
#pragma unroll
              for (int e = 0; e < 8; ++e) u[e] = g * u[e];
              sv = pack8(u);
            }
          } else if (a.state != nullptr && W + (sj - start) >= 0) {
            sv = ldg16(a.state + (static_cast<int64_t>(r) * W + W + (sj - start)) * C + c);
          }
          *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = sv;
        }
      }
    }
  }

  // Requests with no tokens keep their state (tile 0 copies it through).
  if (a.state_out != nullptr && W > 0 && tile == 0) {
    for (int r = 0; r < a.num_reqs; ++r) {
      int64_t s, e;
      request_span(a.qsl, a.num_reqs, T, r, &s, &e);
      if (e != s) continue;
      for (int idx = tid; idx < W * ng; idx += kThreads) {
        const int64_t off = (static_cast<int64_t>(r) * W + idx / ng) * C + c0 + (idx % ng) * 8;
        const uint4 v = a.state ? ldg16(a.state + off) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(a.state_out + off) = v;
      }
    }
  }

  if constexpr (GATED) {
    // No CTA leaves while a peer may still read its partial sums.
    cooperative_groups::this_cluster().sync();
  }
}

// Launch shape: CL CTAs per tile splitting the channels (slices of >= 512
// channels, a multiple of 8), TT tokens per tile so that the grid has at
// least ~3 CTAs per SM. PLE_CONV_TILE / PLE_CONV_SPLIT override the choice
// (launch-shape sweeps).
void pick_conv_shape(int64_t T, int C, int* TT, int* CL) {
  int cl = 8;
  while (cl > 1 && (C % (cl * 8) != 0 || C / cl < 512)) cl >>= 1;
  int tt = 64;
  const int64_t target = 3 * static_cast<int64_t>(num_sms());
  while (tt > 8 && ((T + tt - 1) / tt) * cl < target) tt >>= 1;
  if (const char* e = getenv("PLE_CONV_TILE")) { int v = atoi(e); if (v >= 1 && v <= 256) tt = v; }
  if (const char* e = getenv("PLE_CONV_SPLIT")) {
    int v = atoi(e);
    if (v >= 1 && v <= 8 && C % (v * 8) == 0) cl = v;
  }
  *TT = tt;
  *CL = cl;
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
  pick_conv_shape(T, C, &a.TT, &a.CL);
  a.slice = C / a.CL;
  const ConvSmem L = conv_smem_layout(a.TT, K, dil, a.slice);
  if (L.total > 227 * 1024)
    return fail(PLE_ERR_UNSUPPORTED, "%s: %zu bytes of shared memory needed", name, L.total);
  auto kernel = gated ? conv_kernel<true> : conv_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L.total));
  if (err != cudaSuccess) return check_cuda(err, name);
  const int64_t tiles = (T + a.TT - 1) / a.TT;
  if (tiles * a.CL > 0x7fffffff) return fail(PLE_ERR_UNSUPPORTED, "%s: too many tokens", name);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * a.CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = gated ? a.CL : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kernel, a);
  if (err != cudaSuccess) return check_cuda(err, name);
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
