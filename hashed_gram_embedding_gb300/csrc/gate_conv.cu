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
constexpr int kConvThreads = 512;
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

// gamma_h[c] * gamma_k[c] for 8 channels, from the two bf16 vectors in
// global memory (standalone gate) ...
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

// ... or precomputed once per CTA in shared memory (fused kernel). Both give
// the same float32 products, so the two kernels agree bit for bit.
struct GammaFromShared {
  const float* gg;
  __device__ __forceinline__ void operator()(int c, float out[8]) const {
    const float4 x = *reinterpret_cast<const float4*>(gg + c);
    const float4 y = *reinterpret_cast<const float4*>(gg + c + 4);
    out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
    out[4] = y.x; out[5] = y.y; out[6] = y.z; out[7] = y.w;
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

// Request boundaries of the requests a CTA touches, staged in shared memory
// (falls back to global memory when there are too many).
struct Bounds {
  const int32_t* qsl;    // global
  const int32_t* s;      // shared copy of qsl[r0 .. r0 + n], or nullptr
  int r0, n, num_reqs;
  int64_t T;

  __device__ __forceinline__ int find(int64_t t) const {
    if (s == nullptr) return find_request(qsl, num_reqs, t);
    int lo = 0, hi = n + 1;  // count of staged boundaries <= t
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(s[mid]) <= t) lo = mid + 1; else hi = mid;
    }
    int r = r0 + lo - 1;
    r = r < r0 ? r0 : r;
    return r >= num_reqs ? num_reqs - 1 : r;
  }
  __device__ __forceinline__ void span(int r, int64_t* start, int64_t* end) const {
    if (s == nullptr || r < r0 || r >= r0 + n) {
      request_span(qsl, num_reqs, T, r, start, end);
      return;
    }
    int64_t st = s[r - r0];
    int64_t e = (r + 1 < num_reqs) ? static_cast<int64_t>(s[r + 1 - r0]) : T;
    st = st < 0 ? 0 : (st > T ? T : st);
    e = e < st ? st : (e > T ? T : e);
    *start = st;
    *end = e;
  }
};

// One walker: tokens tt = first, first + d, ... < s1 of the tile (tile-relative),
// for 8 channels c..c+7 of the current window chunk.
template <bool GATED, int K>
struct ConvWalker {
  static __device__ __forceinline__ void load_u(const ConvArgs& a, const uint4* win, const float* g_s,
                                                int vecs, int cv, int c, int64_t j, int64_t start,
                                                int r, int64_t row0, int W, float u[8]) {
    if (j >= start) {
      const int row = static_cast<int>(j - row0);
      unpack8(win[row * vecs + cv], u);
      if constexpr (GATED) {
        const float g = g_s[row];
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = g * u[e];
        unpack8(pack8(u), u);  // u is a bf16 value (a step boundary)
      }
    } else {
      const int64_t hp = W + (j - start);  // history row, oldest first
      uint4 h = make_uint4(0, 0, 0, 0);
      if (a.state != nullptr && hp >= 0)
        h = ldg16(a.state + (static_cast<int64_t>(r) * W + hp) * a.C + c);
      unpack8(h, u);
    }
  }

  static __device__ void run(const ConvArgs& a, const uint4* win, const float* g_s,
                             const float* w_col, int chunk, int vecs, int cv, int c,
                             const int4* tok_s, int64_t t0, int64_t row0, int W, int dil,
                             int first, int s1) {
    if (first >= s1) return;
    float wt[K][8];
    float ring[K][8];  // ring[K-1] = u of the current token, ring[K-1-m] = m*d back
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const float4 w0 = *reinterpret_cast<const float4*>(w_col + i * chunk);
      const float4 w1 = *reinterpret_cast<const float4*>(w_col + i * chunk + 4);
      wt[i][0] = w0.x; wt[i][1] = w0.y; wt[i][2] = w0.z; wt[i][3] = w0.w;
      wt[i][4] = w1.x; wt[i][5] = w1.y; wt[i][6] = w1.z; wt[i][7] = w1.w;
    }
    int cur_start = -1 << 30;  // tile-relative start of the ring's request
    for (int tt = first; tt < s1; tt += dil) {
      const int4 sr = tok_s[tt];  // (start - t0, end - t0, request)
      const int64_t t = t0 + tt;
      const int64_t start = t0 + sr.x;
      if (sr.x != cur_start) {  // first token of the walk or a new request: refill
        cur_start = sr.x;
#pragma unroll
        for (int m = 1; m < K; ++m)
          load_u(a, win, g_s, vecs, cv, c, t - static_cast<int64_t>(m) * dil, start, sr.z, row0, W,
                 ring[K - 1 - m]);
      } else {
#pragma unroll
        for (int i = 0; i + 1 < K; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) ring[i][e] = ring[i + 1][e];
      }
      load_u(a, win, g_s, vecs, cv, c, t, start, sr.z, row0, W, ring[K - 1]);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < K; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wt[i][e], ring[i][e], acc[e]);
      *reinterpret_cast<uint4*>(a.out + t * a.C + c) = pack8(acc);
      // Carry-over: the walker holding a request's last token writes the
      // request's new state (the last W inputs, any residue class).
      if (a.state_out != nullptr && W > 0 && tt == sr.y - 1) {
        for (int jj = 0; jj < W; ++jj) {
          float u[8];
          load_u(a, win, g_s, vecs, cv, c, t - W + 1 + jj, start, sr.z, row0, W, u);
          *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(sr.z) * W + jj) * a.C + c) =
              pack8(u);
        }
      }
    }
  }
};

constexpr int kStagedBounds = 1024;  // request boundaries staged per CTA
constexpr int kMaxTileTokens = 64;   // tokens per CTA (bounds the staged window)

// Shared-memory layout of conv_kernel (byte offsets).
struct ConvLayout {
  size_t gg, bounds, g, tok, w, buf0, buf_bytes, bars, total;
  int rows, chunk;
};

__host__ __device__ inline ConvLayout conv_layout(int C, int W, int tile_tokens, bool gated,
                                                  int chunk) {
  ConvLayout L;
  L.rows = tile_tokens + W;
  L.chunk = chunk;
  size_t off = 0;
  L.gg = off;      off += gated ? static_cast<size_t>(C) * 4 : 0;       // gamma_h * gamma_k
  L.bounds = off;  off += kStagedBounds * 4;                            // query_start_loc slice
  L.g = off;       off += static_cast<size_t>(L.rows) * 4;              // gate scalars
  off = (off + 15) & ~size_t(15);
  L.tok = off;     off += static_cast<size_t>(tile_tokens) * 16;        // per-token (start, end, req)
  L.w = off;       off += static_cast<size_t>(kMaxK) * chunk * 4;       // taps of the chunk, f32
  off = (off + 127) & ~size_t(127);
  L.buf0 = off;
  L.buf_bytes = static_cast<size_t>(L.rows) * chunk * 2;                // one window buffer
  off += 2 * L.buf_bytes;
  off = (off + 7) & ~size_t(7);
  L.bars = off;    off += 16;
  L.total = off;
  return L;
}

// Channel chunk of the staged window: the widest of 512/256/128/64/.../8
// channels dividing C whose two buffers fit next to the rest.
__host__ __device__ inline int conv_chunk(int C, int W, int tile_tokens, bool gated) {
  for (int ch = 512; ch >= 8; ch >>= 1) {
    if (C % ch != 0) continue;
    if (conv_layout(C, W, tile_tokens, gated, ch).total <= 200 * 1024) return ch;
  }
  return 0;
}

template <bool GATED, int K>
__global__ void __launch_bounds__(kConvThreads, 1)
conv_kernel(const __grid_constant__ ConvArgs a, int tile_tokens, int chunk) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int dil = a.dil;
  const int W = (K - 1) * dil;
  const int C = a.C;
  const int64_t T = a.T;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const ConvLayout L = conv_layout(C, W, tile_tokens, GATED, chunk);
  float* gg_s = reinterpret_cast<float*>(smem + L.gg);
  int32_t* qsl_s = reinterpret_cast<int32_t*>(smem + L.bounds);
  float* g_s = reinterpret_cast<float*>(smem + L.g);
  int4* tok_s = reinterpret_cast<int4*>(smem + L.tok);   // (start - t0, end - t0, request) per token
  float* w_s = reinterpret_cast<float*>(smem + L.w);      // [K][chunk]
  const uint32_t bar0 = smem_u32(smem + L.bars);
  auto buffer = [&](int bsel) {
    return reinterpret_cast<uint4*>(smem + L.buf0 + static_cast<size_t>(bsel) * L.buf_bytes);
  };

  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tile_tokens;
  const int64_t t1 = t0 + tile_tokens < T ? t0 + tile_tokens : T;
  const int n_tok = static_cast<int>(t1 - t0);
  const int64_t row0 = t0 - W;              // window row i <-> token row0 + i
  const int vecs = chunk / 8;                // 16-byte vectors per window row
  const int n_chunks = C / chunk;
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const int64_t src_off = GATED ? C : 0;    // v sits after k in kv

  if (blockIdx.x == 0)
    for (int i = tid; i < a.num_reqs + 1; i += kConvThreads)
      check_qsl(a.qsl, a.num_reqs, T, i, a.dev_err);

  // Boundaries of the requests the tile and its halo touch.
  const int r_lo = find_request(a.qsl, a.num_reqs, row0 > 0 ? row0 : 0);
  const int r_hi = find_request(a.qsl, a.num_reqs, t1 - 1);
  const int nb = r_hi - r_lo + 1;
  const bool staged = nb >= 1 && nb + 1 <= kStagedBounds;
  if (staged)
    for (int i = tid; i <= nb; i += kConvThreads)
      qsl_s[i] = (r_lo + i <= a.num_reqs) ? __ldg(a.qsl + r_lo + i) : static_cast<int32_t>(T);
  if constexpr (GATED) {
    for (int c = tid; c < C; c += kConvThreads)
      gg_s[c] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.gamma_h)[c]) *
                __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.gamma_k)[c]);
  }
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const Bounds b{a.qsl, staged ? qsl_s : nullptr, r_lo, nb, a.num_reqs, T};
  for (int i = tid; i < n_tok; i += kConvThreads) {
    const int r = b.find(t0 + i);
    int64_t st, en;
    b.span(r, &st, &en);
    tok_s[i] = make_int4(static_cast<int>(st - t0), static_cast<int>(en - t0), r, 0);
  }
  // Window rows before the start of t0's request belong to other requests.
  int64_t lo, lo_end;
  b.span(b.find(t0), &lo, &lo_end);
  const int i_lo = static_cast<int>(lo > row0 ? lo - row0 : 0);
  const int i_hi = W + n_tok;
  const uint32_t row_bytes = static_cast<uint32_t>(chunk) * 2;

  // Issue the bulk copies of window chunk k (rows [i_lo, i_hi)) into buffer k % 2.
  int issued[2] = {0, 0};  // copies issued into each buffer (uniform over the CTA)
  auto issue = [&](int k) {
    const int bsel = k & 1;
    ++issued[bsel];
    if (warp == 0) {
      const uint32_t bar = bar0 + 8u * bsel;
      if (lane == 0) mbar_arrive_expect_tx(bar, row_bytes * static_cast<uint32_t>(i_hi - i_lo));
      __syncwarp();
      const int c0 = k * chunk;
      for (int i = i_lo + lane; i < i_hi; i += 32)
        bulk_copy_g2s(smem_u32(buffer(bsel)) + static_cast<uint32_t>(i) * row_bytes,
                      a.src + (row0 + i) * src_pitch + src_off + c0, row_bytes, bar);
    }
  };
  issue(0);
  if (n_chunks > 1) issue(1);

  // 1. gate scalars of window rows [i_lo, i_hi), one warp per row (overlaps the copies)
  if constexpr (GATED) {
    const GammaFromShared gamma{gg_s};
    for (int i = i_lo + warp; i < i_hi; i += kConvWarps) {
      const int64_t j = row0 + i;
      const float g = gate_scalar(a.hidden + j * C, a.src + j * src_pitch, gamma, C, a.eps, lane);
      if (lane == 0) {
        g_s[i] = g;
        if (a.gate_out != nullptr && i >= W) a.gate_out[j] = g;
      }
    }
  }
  __syncthreads();

  // 2. per channel chunk: wait for the window, then walkers convolve it.
  //    A walker owns 8 channels, one residue class rho mod d and a segment of
  //    the tile; the taps of y_t sit at t, t-d, ..., t-(K-1)d, all in its own
  //    class, so a ring of K gated values (float32 registers) holds the
  //    dilation window and each gated value is computed once.
  const int per_seg = vecs * dil;
  int segs = kConvThreads / per_seg;
  if (segs < 1) segs = 1;
  const int max_segs = (n_tok + dil - 1) / dil;
  if (segs > max_segs) segs = max_segs > 0 ? max_segs : 1;
  bool ok = true;
  for (int kc = 0; kc < n_chunks && ok; ++kc) {
    const int bsel = kc & 1;
    const uint32_t parity = static_cast<uint32_t>(kc >> 1) & 1u;
    const int c0 = kc * chunk;
    for (int idx = tid; idx < K * chunk; idx += kConvThreads) {
      const int i = idx / chunk;
      const int cc = idx - i * chunk;
      w_s[idx] = __uint_as_float(static_cast<uint32_t>(__ldg(
                     reinterpret_cast<const uint16_t*>(a.w) + static_cast<int64_t>(c0 + cc) * K + i)) << 16);
    }
    ok = mbar_wait(bar0 + 8u * bsel, parity, nullptr);
    if (!ok) {
      if (tid == 0) set_dev_err(a.dev_err, PLE_DEVERR_TIMEOUT);
      break;
    }
    __syncthreads();  // w_s complete (the window is complete per the barrier)
    const uint4* win = buffer(bsel);
    for (int item = tid; item < per_seg * segs; item += kConvThreads) {
      const int cv = item % vecs;
      const int rho = (item / vecs) % dil;
      const int seg = item / per_seg;
      const int c = c0 + cv * 8;
      const int s0 = n_tok * seg / segs;
      const int s1 = n_tok * (seg + 1) / segs;
      ConvWalker<GATED, K>::run(a, win, g_s, w_s + cv * 8, chunk, vecs, cv, c, tok_s, t0, row0, W,
                                dil, s0 + rho, s1);
    }
    __syncthreads();  // every read of this buffer is done
    if (kc + 2 < n_chunks) issue(kc + 2);
  }
  if (!ok) {
    // never leave with copies in flight into this CTA's shared memory: wait
    // (bounded) for the last fill of each buffer
    for (int b2 = 0; b2 < 2; ++b2)
      if (issued[b2] > 0)
        mbar_wait(bar0 + 8u * b2, static_cast<uint32_t>(issued[b2] - 1) & 1u, nullptr);
  }

  // Requests with no tokens keep their state (CTA 0 copies it through).
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    const int ng = C / 8;
    for (int r = 0; r < a.num_reqs; ++r) {
      int64_t s0, e0;
      request_span(a.qsl, a.num_reqs, T, r, &s0, &e0);
      if (e0 != s0) continue;
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

// Tokens per CTA: enough CTAs for every SM, at most kMaxTileTokens.
// PLE_CONV_TILE overrides (launch-shape sweeps).
int conv_tile_tokens(int64_t T) {
  int64_t per = (T + num_sms() - 1) / num_sms();
  if (per < 4) per = 4;
  if (per > kMaxTileTokens) per = kMaxTileTokens;
  if (const char* e = getenv("PLE_CONV_TILE")) {
    const int v = atoi(e);
    if (v >= 1 && v <= kMaxTileTokens) per = v;
  }
  return static_cast<int>(per);
}

template <bool GATED>
ple_status launch_conv(const ConvArgs& a, cudaStream_t stream, const char* name) {
  const int W = (a.K - 1) * a.dil;
  const int tile = conv_tile_tokens(a.T);
  const int chunk = conv_chunk(a.C, W, tile, GATED);
  if (chunk == 0) return fail(PLE_ERR_UNSUPPORTED, "%s: window does not fit in shared memory", name);
  const ConvLayout L = conv_layout(a.C, W, tile, GATED, chunk);
  void (*kernel)(ConvArgs, int, int) = nullptr;
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
                                         static_cast<int>(L.total));
  if (err != cudaSuccess) return check_cuda(err, name);
  const int64_t grid = (a.T + tile - 1) / tile;
  if (grid > 0x7fffffff) return fail(PLE_ERR_UNSUPPORTED, "%s: too many tokens", name);
  kernel<<<static_cast<unsigned>(grid), kConvThreads, L.total, stream>>>(a, tile, chunk);
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
