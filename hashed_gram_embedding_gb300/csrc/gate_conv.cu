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
//   pass 1 (gate_stream_kernel): one warp per token reduces sum h^2, sum k^2
//     and sum h*k*gh*gk over the hidden row; the rows stream into shared
//     memory by bulk async copies, several tokens in flight per warp, one CTA
//     per SM over a contiguous token range. It writes the gate scalar g_t
//     (4 bytes per token); ple_gate's variant also writes u = bf16(g*v).
//   pass 2 (conv_kernel<GATED=true>): a CTA takes a tile of tokens and a
//     256-channel slice, stages its dilation window -- u of the tile and of
//     the (K-1)*d tokens before it -- in shared memory as bf16 (u is a bf16
//     value; 512 bytes per row; for large steps one TMA copy of the raw v
//     rows, then u = bf16(g*v) in place; for small ones per-lane loads),
//     then each lane owns 8 channels (taps in registers as bf16 pairs,
//     float32 accumulators, mixed-precision FMAs).
//     When every token of the tile has all its taps inside its own request,
//     each warp walks a block of tokens along its dilation chains with the
//     K window rows of a token in a register ring (a row is read from shared
//     memory once per chain, not once per tap); otherwise each warp walks
//     tokens one by one, and a request's first (K-1)*d tokens take the taps
//     before its start from the carry-over state. The CTA holding a
//     request's last token writes the request's new state for its channels.
// ple_conv is pass 2 on an ungated input; ple_gate is pass 1 plus u = g*v.
#include "common.cuh"
#include "tma.cuh"

#include <cstdlib>
#include <cstring>

namespace ple {
namespace {

constexpr int kConvThreads = 256;
constexpr int kMaxK = 8;
constexpr int kMaxHalo = 64;
constexpr int kMaxGateC = 16384;  // 8 vectors per thread at 256 threads per token

// u = bf16(g * v) for one bf16 pair word.
__device__ __forceinline__ uint32_t gate2(uint32_t w, float g) {
  return pack2(__fmul_rn(bf_lo(w), g), __fmul_rn(bf_hi(w), g));
}
__device__ __forceinline__ uint4 gate8(uint4 v, float g) {
  return make_uint4(gate2(v.x, g), gate2(v.y, g), gate2(v.z, g), gate2(v.w, g));
}


// ---------------------------------------------------------------------------
// Pass 1: gate scalars (and, for ple_gate, u = bf16(g * v)), streamed.
// One CTA per SM takes a contiguous range of tokens; each warp takes every
// W-th token of it and keeps S tokens in flight: lane 0 bulk-copies the
// token's h row and k row (4C bytes) into one of the warp's S shared-memory
// slots, completing on that slot's mbarrier, so HBM sees W*S*4C bytes of
// requests per SM at once while the warp reduces an earlier slot. Lane l
// owns the 16-byte vectors l, l+32, ... of a row; gamma_h * gamma_k sits in
// shared memory laid out to match. Sums are float pairs (even / odd channel)
// accumulated with two-wide FMAs over the lane's vectors in order, then
// even + odd, then a butterfly over the warp: ple_gate and ple_gate_conv run
// this same kernel, so both produce the same g bit for bit.
// ---------------------------------------------------------------------------
constexpr int kGsMaxWarps = 8;
constexpr size_t kGsSmemBudget = 220 * 1024;
constexpr int kGsChunk = 2048;  // channels of a row per slot (rows stream in chunks)

// Bytes of the gamma-product table: [ceil(nv / 32)][2][32] float4, nv = C / 8
// (whole groups of 32 vectors, so a ragged last group still has its place).
__host__ __device__ inline size_t gate_gg_bytes(int C) {
  return static_cast<size_t>((C / 8 + 31) / 32) * 1024;
}

struct GateStream {
  int warps;     // per CTA
  int slots;     // per warp
  size_t gg_bytes, slot_bytes, smem;
};

GateStream gate_stream_shape(int C) {
  GateStream g{};
  g.gg_bytes = gate_gg_bytes(C);
  g.slot_bytes = static_cast<size_t>(C < kGsChunk ? C : kGsChunk) * 4;  // h and k chunk, bf16
  for (int slots = 3; slots >= 2; --slots) {
    const size_t per_warp = slots * (g.slot_bytes + 8);
    if (g.gg_bytes + per_warp > kGsSmemBudget) continue;
    size_t warps = (kGsSmemBudget - g.gg_bytes) / per_warp;
    if (warps > kGsMaxWarps) warps = kGsMaxWarps;
    g.warps = static_cast<int>(warps);
    g.slots = slots;
    g.smem = g.gg_bytes + warps * per_warp;
    return g;
  }
  return g;  // warps == 0: too large
}

template <bool WRITE_U>
__global__ void __launch_bounds__(kGsMaxWarps * 32)
gate_stream_kernel(const ple_bf16_t* __restrict__ hidden, const ple_bf16_t* __restrict__ kv,
                   const ple_bf16_t* __restrict__ gamma_h, const ple_bf16_t* __restrict__ gamma_k,
                   float eps, int64_t T, int C, int slots, ple_bf16_t* __restrict__ u_out,
                   float* __restrict__ gate_out, int32_t* dev_err) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int warps = blockDim.x >> 5;
  const int nv = C >> 3;
  const size_t gg_bytes = gate_gg_bytes(C);
  const int CC = C < kGsChunk ? C : kGsChunk;  // channels per chunk
  const int nch = (C + CC - 1) / CC;           // chunks per row
  const size_t slot_bytes = static_cast<size_t>(CC) * 4;
  float4* gg4 = reinterpret_cast<float4*>(smem);  // [nv/32][2][32]
  uint8_t* slot0 = smem + gg_bytes + static_cast<size_t>(warp) * slots * slot_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + gg_bytes +
                                               static_cast<size_t>(warps) * slots * slot_bytes);
  const uint32_t bar0 = smem_u32(bars + warp * slots);

  if (tid == 0) {
    for (int i = 0; i < warps * slots; ++i) mbar_init(smem_u32(bars + i), 1);
    mbar_fence_init();
  }
  pdl_wait();  // k comes from the previous kernel
  pdl_trigger();
  for (int v = tid; v < nv; v += blockDim.x) {
    const uint4 a = ldg16(gamma_h + v * 8);
    const uint4 b = ldg16(gamma_k + v * 8);
    float fa[8], fb[8];
    unpack8(a, fa);
    unpack8(b, fb);
    gg4[((v >> 5) * 2) * 32 + (v & 31)] =
        make_float4(fa[0] * fb[0], fa[1] * fb[1], fa[2] * fb[2], fa[3] * fb[3]);
    gg4[((v >> 5) * 2 + 1) * 32 + (v & 31)] =
        make_float4(fa[4] * fb[4], fa[5] * fb[5], fa[6] * fb[6], fa[7] * fb[7]);
  }
  __syncthreads();

  // items of this warp: (token k, chunk j), m = k * nch + j
  const int64_t ta = T * blockIdx.x / gridDim.x;
  const int64_t tb = T * (blockIdx.x + 1) / gridDim.x;
  const int64_t n_tok = tb - ta > warp ? (tb - ta - warp + warps - 1) / warps : 0;
  const int64_t n_items = n_tok * nch;
  auto token = [&](int64_t k) { return ta + warp + k * warps; };
  auto chunk_ch = [&](int j) { return C - j * CC < CC ? C - j * CC : CC; };
  auto issue = [&](int64_t m) {  // lane 0 only
    const int64_t t = token(m / nch);
    const int j = static_cast<int>(m % nch);
    const uint32_t bytes = static_cast<uint32_t>(chunk_ch(j)) * 2;
    const int sl = static_cast<int>(m % slots);
    const uint32_t bar = bar0 + 8u * sl;
    const uint32_t dst = smem_u32(slot0 + sl * slot_bytes);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_copy_g2s(dst, hidden + t * C + j * CC, bytes, bar);
    bulk_copy_g2s(dst + static_cast<uint32_t>(CC) * 2, kv + t * 2 * C + j * CC, bytes, bar);
  };
  if (lane == 0)
    for (int64_t m = 0; m < n_items && m < slots; ++m) issue(m);

  uint64_t sh2 = 0, sk2 = 0, sd2 = 0;  // +0.0f pairs, over a token's chunks
  int64_t m = 0;
  for (; m < n_items; ++m) {
    const int sl = static_cast<int>(m % slots);
    const uint32_t parity = static_cast<uint32_t>((m / slots) & 1);
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * sl, parity, nullptr))) {
      if (lane == 0) set_dev_err(dev_err, PLE_DEVERR_TIMEOUT);
      break;
    }
    const int j = static_cast<int>(m % nch);
    const int nvc = chunk_ch(j) >> 3;
    const int v0 = j * (CC >> 3);  // first vector of the chunk (a multiple of 32 or 0)
    const uint4* h4 = reinterpret_cast<const uint4*>(slot0 + sl * slot_bytes);
    const uint4* k4 = reinterpret_cast<const uint4*>(slot0 + sl * slot_bytes + static_cast<size_t>(CC) * 2);
    for (int vl = lane; vl < nvc; vl += 32) {
      const int i = (v0 + vl) >> 5;  // group of 32 vectors of the row
      const uint4 hv = h4[vl];
      const uint4 kk = k4[vl];
      const float4 g0 = gg4[(i * 2) * 32 + lane];
      const float4 g1 = gg4[(i * 2 + 1) * 32 + lane];
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
      const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w};
      const uint64_t gp[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint64_t h2 = f2(bf_lo(hw[p]), bf_hi(hw[p]));
        const uint64_t k2 = f2(bf_lo(kw[p]), bf_hi(kw[p]));
        sh2 = f2_fma(h2, h2, sh2);
        sk2 = f2_fma(k2, k2, sk2);
        sd2 = f2_fma(f2_mul(h2, k2), gp[p], sd2);
      }
    }
    __syncwarp();
    if (lane == 0 && m + slots < n_items) {
      // the slot was read through the generic proxy; order that before the
      // bulk copy (async proxy) that refills it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(m + slots);
    }
    if (j != nch - 1) continue;
    float a0, a1, b0, b1, d0, d1;
    f2_split(sh2, a0, a1);
    f2_split(sk2, b0, b1);
    f2_split(sd2, d0, d1);
    sh2 = sk2 = sd2 = 0;
    const float g = gate_of(warp_sum(a0 + a1), warp_sum(b0 + b1), warp_sum(d0 + d1), C, eps);
    const int64_t t = token(m / nch);
    if (lane == 0 && gate_out != nullptr) gate_out[t] = g;
    if constexpr (WRITE_U) {
      const ple_bf16_t* v_row = kv + t * 2 * C + C;
      for (int v = lane; v < nv; v += 32)
        *reinterpret_cast<uint4*>(u_out + t * C + v * 8) = gate8(ldg16(v_row + v * 8), g);
    }
  }
  // after a timeout: never leave with a copy in flight into this warp's slots
  if (lane == 0)
    for (int64_t q = m; q < n_items && q < m + slots; ++q)
      mbar_wait(bar0 + 8u * static_cast<uint32_t>(q % slots),
                static_cast<uint32_t>((q / slots) & 1), nullptr);
}

template <bool WRITE_U>
ple_status gate_pass(const ple_bf16_t* hidden, const ple_bf16_t* kv, const ple_bf16_t* gamma_h,
                     const ple_bf16_t* gamma_k, float eps, int64_t T, int C, ple_bf16_t* u_out,
                     float* gate_out, int32_t* dev_err, cudaStream_t stream, const char* name) {
  const GateStream gs = gate_stream_shape(C);
  if (gs.warps == 0 || C > kMaxGateC)
    return fail(PLE_ERR_UNSUPPORTED, "%s: hidden_size %d above %d", name, C, kMaxGateC);
  cudaError_t err = cudaFuncSetAttribute(gate_stream_kernel<WRITE_U>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gs.smem));
  if (err != cudaSuccess) return check_cuda(err, name);
  const int64_t grid = T < num_sms() ? T : num_sms();
  err = launch_kernel(gate_stream_kernel<WRITE_U>, dim3(static_cast<unsigned>(grid)),
                      dim3(gs.warps * 32), gs.smem, stream, 1, hidden, kv, gamma_h, gamma_k, eps,
                      T, C, gs.slots, u_out, gate_out, dev_err);
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}

// ---------------------------------------------------------------------------
// ple_conv (GATED = false, input x) and ple_gate_conv (GATED = true).
// ---------------------------------------------------------------------------
struct ConvArgs {
  const ple_bf16_t* src;      // kv (gated: v is its second half) or x
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
  int32_t* dev_err;
};

constexpr int kConvSlice = 256;  // channels per CTA (8 per lane)

// Shared memory of one conv CTA: the bf16 window (rows x 512 bytes: lane l
// holds channels 8l..8l+7 as one 16-byte vector, so a warp's accesses to a
// row are contiguous), then per-token and per-request integers.
struct ConvSmem {
  uint4* win;
  int* tok_start;  // [tile] start of the token's request, relative to t0
  int* tok_req;    // [tile] the token's request
  int* req_s;      // [tile] requests overlapping the tile: start, end (rel.), index
  int* req_e;
  int* req_r;
  int* counts;     // [0] requests listed, [1] requests ending in the tile
  int* end_k;      // [tile] list positions of the requests ending in the tile
  float* gs;       // [tile + W] gate scalars of the window rows (TMA staging)
  uint64_t* bar;   // the window copy's mbarrier (TMA staging)
};

// Window, lists, gate scalars and mbarrier, plus room to align the window
// to 128 bytes (a TMA destination).
__host__ __device__ inline size_t conv_smem_bytes(int tile, int W) {
  return static_cast<size_t>(tile + W) * kConvSlice * 2 + static_cast<size_t>(tile) * 6 * 4 + 16 +
         static_cast<size_t>(tile + W) * 4 + 8 + 128;
}

__device__ __forceinline__ ConvSmem conv_smem(uint8_t* base, int tile, int W) {
  ConvSmem s;
  s.win = reinterpret_cast<uint4*>(base);
  int* p = reinterpret_cast<int*>(base + static_cast<size_t>(tile + W) * kConvSlice * 2);
  s.tok_start = p;
  s.tok_req = p + tile;
  s.req_s = p + 2 * tile;
  s.req_e = p + 3 * tile;
  s.req_r = p + 4 * tile;
  s.end_k = p + 5 * tile;
  s.counts = p + 6 * tile;
  s.gs = reinterpret_cast<float*>(p + 6 * tile + 4);
  s.bar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(s.gs + tile + W) + 7) & ~static_cast<uintptr_t>(7));
  return s;
}

// Requests overlapping [t0, t0 + n_tok), found by warp 0: a 32-way search
// for the request of t0, then the following qsl entries 32 at a time. Spans
// follow request_span (clamped; the last request ends at T). With a valid
// qsl there are at most n_tok non-empty overlapping requests; extra entries
// (possible only for an invalid qsl) are dropped.
__device__ void find_tile_requests(const int32_t* __restrict__ qsl, int R, int64_t T, int64_t t0,
                                   int n_tok, int cap, ConvSmem s, int lane) {
  // cnt = number of entries qsl[0..R] <= t0 for a non-decreasing qsl
  int lo = 0, hi = R + 1;
  while (lo < hi) {
    const int step = (hi - lo + 31) >> 5;
    const int p = lo + lane * step;
    const bool le = p < hi && static_cast<int64_t>(__ldg(qsl + p)) <= t0;
    const int k = __popc(__ballot_sync(0xffffffffu, le));
    if (k == 0) break;
    const int nlo = lo + (k - 1) * step + 1;
    hi = min(lo + k * step, hi);
    lo = nlo;
  }
  int r = lo - 1;
  r = r < 0 ? 0 : (r >= R ? R - 1 : r);
  int listed = 0, ending = 0;
  const int64_t t1 = t0 + n_tok;
  for (; r < R; r += 32) {
    const int rr = r + lane;
    bool take = false, beyond = false;
    int64_t st = 0, en = 0;
    if (rr < R) {
      request_span(qsl, R, T, rr, &st, &en);
      take = en > st && st < t1 && en > t0;
      beyond = st >= t1;
    }
    const unsigned m = __ballot_sync(0xffffffffu, take);
    const int pos = listed + __popc(m & ((1u << lane) - 1));
    if (take && pos < cap) {
      s.req_s[pos] = static_cast<int>(st - t0);
      s.req_e[pos] = static_cast<int>(en - t0);
      s.req_r[pos] = rr;
    }
    const bool ends = take && pos < cap && en <= t1;
    const unsigned me = __ballot_sync(0xffffffffu, ends);
    if (ends) s.end_k[ending + __popc(me & ((1u << lane) - 1))] = pos;
    listed = min(listed + __popc(m), cap);
    ending = min(ending + __popc(me), cap);
    if (__ballot_sync(0xffffffffu, beyond) != 0u) break;
  }
  if (lane == 0) {
    s.counts[0] = listed;
    s.counts[1] = ending;
  }
}

// CTAs per SM the register cap allows. Per-lane staging: 3 for K <= 4 (80
// registers: 10 staged rows in flight per lane; a 4-CTA cap of 64 registers
// measured slower), 2 above (the taps and the register ring of K rows grow
// with K). TMA staging holds no rows in registers: 4 for K <= 4 (64
// registers, no spills; the shared memory of an 88-token tile).
__host__ __device__ constexpr int conv_ctas_per_sm(int K, bool tma) {
  return K <= 4 ? (tma ? 4 : 3) : 2;
}
template <bool GATED, int K, bool TMA>
__global__ void __launch_bounds__(kConvThreads, conv_ctas_per_sm(K, TMA))
conv_kernel(const __grid_constant__ ConvArgs a, const float* __restrict__ g, int tile_tokens,
            const __grid_constant__ CUtensorMap map_src, int tma_col0) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const int dil = a.dil;
  const int W = (K - 1) * dil;
  const int C = a.C;
  const int R = a.num_reqs;
  const int64_t T = a.T;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tile_tokens;
  const int n_tok = static_cast<int>((t0 + tile_tokens < T ? t0 + tile_tokens : T) - t0);
  const int c0 = blockIdx.y * kConvSlice;
  const int c = c0 + lane * 8;
  const bool active = c < C;  // lanes past the last channel only help with bookkeeping
  const ConvSmem s = conv_smem(smem, tile_tokens, W);
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const ple_bf16_t* src = a.src + (GATED ? C : 0) + c;
  constexpr bool use_tma = TMA;
  const uint32_t bar = smem_u32(s.bar);
  if (use_tma && tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  if (use_tma) __syncthreads();
  pdl_wait();  // v and g come from the previous kernels
  pdl_trigger();

  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = tid; i < R + 1; i += kConvThreads) check_qsl(a.qsl, R, T, i, a.dev_err);

  if constexpr (TMA) {
    // One TMA copy of the window (rows t0 - W .. t0 + tile - 1 of the slice,
    // 512 bytes each; rows outside [0, T) read as zeros) while the gate
    // scalars of its rows go to shared memory and warp 0 finds the tile's
    // requests; then each warp forms u = bf16(g * v) in place for every 8th
    // row (gated).
    const int rows = tile_tokens + W;
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows) * kConvSlice * 2);
      tma_load_2d(smem_u32(s.win), &map_src, bar, tma_col0 + c0, static_cast<int>(t0 - W));
    }
    if constexpr (GATED) {
      for (int i = tid; i < rows; i += kConvThreads) {
        const int64_t tok = t0 - W + i;
        s.gs[i] = tok >= 0 && tok < T ? __ldg(g + tok) : 0.f;
      }
    }
    if (warp == 0) find_tile_requests(a.qsl, R, T, t0, n_tok, tile_tokens, s, lane);
    if (!__syncthreads_and(mbar_wait(bar, 0, nullptr))) {
      // not within the wait limit: report, and do not leave with the copy in flight
      if (tid == 0) {
        set_dev_err(a.dev_err, PLE_DEVERR_TIMEOUT);
        mbar_wait(bar, 0, nullptr);
      }
      __syncthreads();
      return;
    }
    if constexpr (GATED) {
      __syncthreads();  // the gate scalars
      if (active) {
        for (int i = warp; i < rows; i += kConvThreads / 32) {
          const float gx = s.gs[i];
          const uint4 v = s.win[i * 32 + lane];
          const uint64_t gg = f2(gx, gx);
          uint32_t u4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            float lo, hi;
            f2_split(f2_mul(f2(bf_lo(u4[p]), bf_hi(u4[p])), gg), lo, hi);
            u4[p] = pack2(lo, hi);  // u = bf16(g * v)
          }
          s.win[i * 32 + lane] = make_uint4(u4[0], u4[1], u4[2], u4[3]);
        }
      }
    }
  } else {
    // Window row i <-> token t0 - W + i (rows of tokens before 0 are not
    // loaded; rows of an earlier request are loaded but never read). Each warp
    // takes every 8th row, kBatch rows' loads in flight per lane at a time (one
    // batch covers a 64-token tile and its halo, two a 112-token tile); warp 0
    // searches the tile's requests while its first batch is in flight.
    {
      constexpr int kWarps = kConvThreads / 32;
      constexpr int kBatch = 10;
      const int i0 = t0 >= W ? 0 : static_cast<int>(W - t0);
      const int rows = n_tok + W;
      uint4 v[kBatch];
      float gv[kBatch];
      auto load = [&](int first) {
  #pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = first + q * kWarps;
          v[q] = make_uint4(0, 0, 0, 0);
          gv[q] = 0.f;
          if (active && i < rows) {
            const int64_t tok = t0 - W + i;
            v[q] = ldg16(src + tok * src_pitch);
            if constexpr (GATED) gv[q] = __ldg(g + tok);
          }
        }
      };
      auto stage = [&](int first) {
  #pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = first + q * kWarps;
          if (active && i < rows) {
            if constexpr (GATED) {
              const uint64_t gg = f2(gv[q], gv[q]);
              uint32_t u4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
  #pragma unroll
              for (int p = 0; p < 4; ++p) {
                float lo, hi;
                f2_split(f2_mul(f2(bf_lo(u4[p]), bf_hi(u4[p])), gg), lo, hi);
                u4[p] = pack2(lo, hi);  // u = bf16(g * v)
              }
              s.win[i * 32 + lane] = make_uint4(u4[0], u4[1], u4[2], u4[3]);
            } else {
              s.win[i * 32 + lane] = v[q];
            }
          }
        }
      };
      int first = i0 + warp;
      load(first);
      if (warp == 0) find_tile_requests(a.qsl, R, T, t0, n_tok, tile_tokens, s, lane);
      stage(first);
      for (first += kWarps * kBatch; first < rows; first += kWarps * kBatch) {
        load(first);
        stage(first);
      }
    }
  }
  __syncthreads();

  // request of every tile token (binary search over the listed starts)
  const int listed = s.counts[0];
  int all_fast = 1;  // every token's taps inside its own request
  for (int tt = tid; tt < n_tok; tt += kConvThreads) {
    int lo = 0, hi = listed;  // last k with req_s[k] <= tt
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s.req_s[mid] <= tt) lo = mid + 1; else hi = mid;
    }
    const int k = lo - 1;
    if (k >= 0 && tt < s.req_e[k]) {
      s.tok_start[tt] = s.req_s[k];
      s.tok_req[tt] = s.req_r[k];
    } else {  // only for an invalid qsl: no history
      s.tok_start[tt] = tt;
      s.tok_req[tt] = 0;
    }
    all_fast &= (tt - W >= s.tok_start[tt]) ? 1 : 0;
  }
  all_fast = __syncthreads_and(all_fast);

  // requests with no tokens keep their state (copied by the first token
  // tile; every lane of a warp takes part in the scan)
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    for (int base = warp * 32; base < R; base += kConvThreads) {
      bool empty = false;
      if (base + lane < R) {
        int64_t s0, e0;
        request_span(a.qsl, R, T, base + lane, &s0, &e0);
        empty = e0 == s0;
      }
      unsigned m = __ballot_sync(0xffffffffu, empty);
      while (m != 0u && active) {
        const int r = base + __ffs(m) - 1;
        m &= m - 1;
        for (int jj = 0; jj < W; ++jj) {
          const int64_t off = (static_cast<int64_t>(r) * W + jj) * C + c;
          const uint4 v = a.state ? ldg16(a.state + off) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(a.state_out + off) = v;
        }
      }
    }
  }
  if (!active) return;

  // taps of this lane's 8 channels: w[c..c+7][0..K-1] is 8*K contiguous bf16
  // (K 16-byte loads), regrouped as bf16 pair words wt[tap][pair] (channels
  // 2*pair and 2*pair + 1, the layout of a window word)
  uint32_t wt[K][4];
  {
    uint32_t h[8 * K];  // flat [8][K] bf16 values, one per word
    const uint4* wv = reinterpret_cast<const uint4*>(a.w + static_cast<int64_t>(c) * K);
#pragma unroll
    for (int q = 0; q < K; ++q) {
      const uint4 b = __ldg(wv + q);
      const uint32_t words[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[8 * q + 2 * e] = words[e] & 0xffffu;
        h[8 * q + 2 * e + 1] = words[e] >> 16;
      }
    }
#pragma unroll
    for (int i = 0; i < K; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) wt[i][p] = h[(2 * p) * K + i] | (h[(2 * p + 1) * K + i] << 16);
  }

  // acc[0..7] += taps of tap i times the 8 channels of a bf16 window word
  auto tap = [&](int i, uint4 b, float (&acc)[8]) {
    bf2_fma(wt[i][0], b.x, acc[0], acc[1]);
    bf2_fma(wt[i][1], b.y, acc[2], acc[3]);
    bf2_fma(wt[i][2], b.z, acc[4], acc[5]);
    bf2_fma(wt[i][3], b.w, acc[6], acc[7]);
  };
  auto store = [&](int64_t tok, const float (&acc)[8]) {
    *reinterpret_cast<uint4*>(a.out + tok * C + c) =
        make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                   pack2(acc[6], acc[7]));
  };
  if (all_fast) {
    // each warp takes a contiguous block of tokens and walks it along its
    // dil chains (tokens tt, tt + d, tt + 2d, ...): consecutive tokens of a
    // chain share K - 1 of their K window rows, so the rows stay in a
    // register ring and each is read from shared memory once per chain
    // (the ring is indexed at compile time: the walk is unrolled by K)
    constexpr int kWarps = kConvThreads / 32;
    const int per = (n_tok + kWarps - 1) / kWarps;
    const int b0 = warp * per;
    const int b1 = min(n_tok, b0 + per);
    for (int rho = 0; rho < dil && b0 + rho < b1; ++rho) {
      int tt = b0 + rho;
      uint4 ring[K];
#pragma unroll
      for (int i = 0; i < K - 1; ++i) ring[i] = s.win[(tt + i * dil) * 32 + lane];
      bool more = true;
      while (more) {
#pragma unroll
        for (int u = 0; u < K; ++u) {
          if (more) {
            ring[(u + K - 1) % K] = s.win[(tt + W) * 32 + lane];  // tap K-1: the token itself
            float acc[8] = {};
#pragma unroll
            for (int i = 0; i < K; ++i) tap(i, ring[(u + i) % K], acc);
            store(t0 + tt, acc);
            tt += dil;
            more = tt < b1;
          }
        }
      }
    }
  } else
  for (int tt = warp; tt < n_tok; tt += kConvThreads / 32) {
    const int st = s.tok_start[tt];
    float acc[8] = {};  // +0.0f
    if (tt - W >= st) {
      // all taps inside the request: window rows tt, tt + d, ..., tt + W
#pragma unroll
      for (int i = 0; i < K; ++i) tap(i, s.win[(tt + i * dil) * 32 + lane], acc);
    } else {
      // a request's first W tokens: taps before its start come from the
      // carry-over state (zeros without one); all state loads first
      const int r = s.tok_req[tt];
      uint4 hist[K];
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j = tt - (K - 1 - i) * dil;
        hist[i] = make_uint4(0, 0, 0, 0);
        if (j < st && a.state != nullptr)
          hist[i] = ldg16(a.state + (static_cast<int64_t>(r) * W + (W + j - st)) * C + c);
      }
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j = tt - (K - 1 - i) * dil;
        tap(i, j >= st ? s.win[(tt + i * dil) * 32 + lane] : hist[i], acc);
      }
    }
    store(t0 + tt, acc);
  }

  if (a.state_out == nullptr || W == 0) return;
  // new state of the requests ending in this tile: their last W virtual rows
  const int ending = s.counts[1];
  for (int q = warp; q < ending * W; q += kConvThreads / 32) {
    const int kk = s.end_k[q / W];
    const int jj = q % W;
    const int st = s.req_s[kk];
    const int r = s.req_r[kk];
    const int sj = s.req_e[kk] - W + jj;  // token of state row jj, relative to t0
    uint4 u = make_uint4(0, 0, 0, 0);
    if (sj >= st) {
      u = s.win[(sj + W) * 32 + lane];
    } else if (a.state != nullptr) {
      u = ldg16(a.state + (static_cast<int64_t>(r) * W + (W + sj - st)) * C + c);
    }
    *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = u;
  }
}

// ---------------------------------------------------------------------------
// Streaming conv pass: one CTA per (token range, 256-channel slice), two per
// SM. The CTA walks its range in chunks of CH >= (K-1)*d tokens. Thread 0
// bulk-copies each chunk's rows of the slice (512 bytes each) into one of
// three raw shared-memory slots, two chunks ahead of the one being computed;
// all warps then convert the chunk into a float32 ring of CH + (K-1)*d rows
// (gated: u = bf16(g * v)), which still holds the (K-1)*d rows before the
// chunk, and compute the chunk's outputs from the ring exactly as the tiled
// kernel does (same taps, same FMA order, same bits). Chunk 0 is the halo:
// the (K-1)*d rows before the range.
// ---------------------------------------------------------------------------
constexpr int kCsSlots = 3;

__host__ __device__ inline int conv_stream_chunk(int W) { return W > 32 ? W : 32; }

__host__ __device__ inline size_t conv_stream_smem(int CH, int W) {
  return static_cast<size_t>(CH + W) * kConvSlice * 4           // float32 ring
         + static_cast<size_t>(kCsSlots) * CH * kConvSlice * 2  // raw slots
         + 64                                                   // mbarriers
         + static_cast<size_t>(CH) * 6 * 4 + 16;                // request lists
}

template <bool GATED, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_stream_kernel(const __grid_constant__ ConvArgs a, const float* __restrict__ g, int CH) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int dil = a.dil;
  const int W = (K - 1) * dil;
  const int C = a.C;
  const int R = a.num_reqs;
  const int64_t T = a.T;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  constexpr int kWarps = kConvThreads / 32;
  const int c0 = blockIdx.y * kConvSlice;
  const int slice_ch = C - c0 < kConvSlice ? C - c0 : kConvSlice;
  const uint32_t row_bytes = static_cast<uint32_t>(slice_ch) * 2;
  const int c = c0 + lane * 8;
  const bool active = c < C;
  const int NW = CH + W;  // ring rows
  const int64_t ta = T * blockIdx.x / gridDim.x;
  const int64_t tb = T * (blockIdx.x + 1) / gridDim.x;
  const int nq = static_cast<int>((tb - ta + CH - 1) / CH);  // token chunks; chunk 0 = halo

  float4* ring = reinterpret_cast<float4*>(smem);  // [NW][2][32]
  uint8_t* raw = smem + static_cast<size_t>(NW) * kConvSlice * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + static_cast<size_t>(kCsSlots) * CH * kConvSlice * 2);
  ConvSmem sm;
  {
    int* p = reinterpret_cast<int*>(bars + 8);
    sm.win = nullptr;
    sm.tok_start = nullptr;
    sm.tok_req = nullptr;
    sm.req_s = p;
    sm.req_e = p + CH;
    sm.req_r = p + 2 * CH;
    sm.end_k = p + 3 * CH;
    sm.counts = p + 4 * CH;
  }
  const int64_t src_pitch = GATED ? 2 * static_cast<int64_t>(C) : C;
  const ple_bf16_t* src_slice = a.src + (GATED ? C : 0) + c0;

  if (tid == 0) {
    for (int i = 0; i < kCsSlots; ++i) mbar_init(smem_u32(bars + i), 1);
    mbar_fence_init();
  }
  pdl_wait();  // v and g come from the previous kernels
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = tid; i < R + 1; i += kConvThreads) check_qsl(a.qsl, R, T, i, a.dev_err);
  __syncthreads();

  // rows of chunk q: [first, first + count); chunk 0 is the halo before ta
  auto chunk_first = [&](int q) { return q == 0 ? ta - W : ta + static_cast<int64_t>(q - 1) * CH; };
  auto chunk_count = [&](int q) -> int {
    if (q == 0) return W;
    const int64_t f = ta + static_cast<int64_t>(q - 1) * CH;
    return static_cast<int>(tb - f < CH ? tb - f : CH);
  };
  auto issue = [&](int q) {  // thread 0
    const int sl = q % kCsSlots;
    const uint32_t bar = smem_u32(bars + sl);
    const int64_t first = chunk_first(q);
    const int count = chunk_count(q);
    const int skip = first < 0 ? static_cast<int>(-first) : 0;  // rows before token 0
    const int n = count > skip ? count - skip : 0;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * row_bytes);
    const uint32_t dst = smem_u32(raw + static_cast<size_t>(sl) * CH * kConvSlice * 2);
    for (int r = skip; r < count; ++r)
      bulk_copy_g2s(dst + static_cast<uint32_t>(r) * kConvSlice * 2,
                    src_slice + (first + r) * src_pitch, row_bytes, bar);
  };
  if (tid == 0)
    for (int q = 0; q <= nq && q < kCsSlots; ++q) issue(q);

  // requests with no tokens keep their state (copied by the first range)
  if (a.state_out != nullptr && W > 0 && blockIdx.x == 0) {
    for (int base = warp * 32; base < R; base += kConvThreads) {
      bool empty = false;
      if (base + lane < R) {
        int64_t s0, e0;
        request_span(a.qsl, R, T, base + lane, &s0, &e0);
        empty = e0 == s0;
      }
      unsigned m = __ballot_sync(0xffffffffu, empty);
      while (m != 0u && active) {
        const int r = base + __ffs(m) - 1;
        m &= m - 1;
        for (int jj = 0; jj < W; ++jj) {
          const int64_t off = (static_cast<int64_t>(r) * W + jj) * C + c;
          const uint4 v = a.state ? ldg16(a.state + off) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(a.state_out + off) = v;
        }
      }
    }
  }

  // taps of this lane's 8 channels as float pairs wt[tap][pair]
  uint64_t wt[K][4];
  {
    float wf[K][8];
#pragma unroll
    for (int q = 0; q < K; ++q) {
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (active)
        unpack8(__ldg(reinterpret_cast<const uint4*>(a.w + static_cast<int64_t>(c) * K) + q), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int flat = 8 * q + e;
        wf[flat % K][flat / K] = f[e];
      }
    }
#pragma unroll
    for (int i = 0; i < K; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) wt[i][p] = f2(wf[i][2 * p], wf[i][2 * p + 1]);
  }
  const ulonglong2* ring2 = reinterpret_cast<const ulonglong2*>(ring);
  // The ring holds token ta - W + i at row i mod NW; row of chunk q's first
  // token, and a row a few positions on (less than NW) with one wrap.
  auto chunk_row0 = [&](int q) { return q == 0 ? 0 : static_cast<int>((W + static_cast<int64_t>(q - 1) * CH) % NW); };
  auto wrap = [&](int row) { return row >= NW ? row - NW : row; };

  int q = 0;
  for (; q <= nq; ++q) {
    const int sl = q % kCsSlots;
    const uint32_t parity = static_cast<uint32_t>((q / kCsSlots) & 1);
    const bool ok = mbar_wait(smem_u32(bars + sl), parity, nullptr);
    // B1: every warp is done with chunk q-1 (its ring rows may be reused)
    if (__syncthreads_or(!ok)) {
      if (tid == 0) set_dev_err(a.dev_err, PLE_DEVERR_TIMEOUT);
      break;
    }
    const int64_t first = chunk_first(q);
    const int count = chunk_count(q);
    const int row0 = chunk_row0(q);
    if (q > 0 && warp == 0) find_tile_requests(a.qsl, R, T, first, count, CH, sm, lane);
    // convert the chunk's rows into the ring
    if (active) {
      const uint8_t* slot = raw + static_cast<size_t>(sl) * CH * kConvSlice * 2;
      for (int r = warp; r < count; r += kWarps) {
        const int64_t tok = first + r;
        if (tok < 0) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(slot + static_cast<size_t>(r) * kConvSlice * 2 + lane * 16);
        float f[8];
        if constexpr (GATED) {
          const float gx = __ldg(g + tok);
          const uint64_t gg = f2(gx, gx);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            float lo, hi;
            f2_split(f2_mul(f2(bf_lo(w4[p]), bf_hi(w4[p])), gg), lo, hi);
            const uint32_t u = pack2(lo, hi);  // round to bf16
            f[2 * p] = bf_lo(u);
            f[2 * p + 1] = bf_hi(u);
          }
        } else {
          unpack8(v, f);
        }
        const int rr = wrap(row0 + r);
        ring[(rr * 2) * 32 + lane] = make_float4(f[0], f[1], f[2], f[3]);
        ring[(rr * 2 + 1) * 32 + lane] = make_float4(f[4], f[5], f[6], f[7]);
      }
    }
    __syncthreads();  // B2: ring rows and request lists ready; raw slot free
    if (tid == 0 && q + kCsSlots <= nq) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(q + kCsSlots);
    }
    if (q == 0 || !active) continue;

    const int listed = sm.counts[0];
    for (int tt = warp; tt < count; tt += kWarps) {
      // the token's request: last listed start <= tt
      int lo = 0, hi = listed;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sm.req_s[mid] <= tt) lo = mid + 1; else hi = mid;
      }
      const int k = lo - 1;
      int st = tt, r = 0;  // (invalid qsl only: no history)
      if (k >= 0 && tt < sm.req_e[k]) {
        st = sm.req_s[k];
        r = sm.req_r[k];
      }
      const int64_t t = first + tt;
      const int p0 = wrap(row0 + tt);
      uint64_t acc[4] = {0, 0, 0, 0};
      if (tt - W >= st) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
          int row = p0 - (K - 1 - i) * dil;
          if (row < 0) row += NW;
          const ulonglong2 x0 = ring2[(row * 2) * 32 + lane];
          const ulonglong2 x1 = ring2[(row * 2 + 1) * 32 + lane];
          acc[0] = f2_fma(wt[i][0], x0.x, acc[0]);
          acc[1] = f2_fma(wt[i][1], x0.y, acc[1]);
          acc[2] = f2_fma(wt[i][2], x1.x, acc[2]);
          acc[3] = f2_fma(wt[i][3], x1.y, acc[3]);
        }
      } else {
        uint4 hist[K];
#pragma unroll
        for (int i = 0; i < K; ++i) {
          const int j = tt - (K - 1 - i) * dil;
          hist[i] = make_uint4(0, 0, 0, 0);
          if (j < st && a.state != nullptr)
            hist[i] = ldg16(a.state + (static_cast<int64_t>(r) * W + (W + j - st)) * C + c);
        }
#pragma unroll
        for (int i = 0; i < K; ++i) {
          const int j = tt - (K - 1 - i) * dil;
          uint64_t x[4];
          if (j >= st) {
            int row = p0 - (K - 1 - i) * dil;
            if (row < 0) row += NW;
            const ulonglong2 x0 = ring2[(row * 2) * 32 + lane];
            const ulonglong2 x1 = ring2[(row * 2 + 1) * 32 + lane];
            x[0] = x0.x; x[1] = x0.y; x[2] = x1.x; x[3] = x1.y;
          } else {
            x[0] = f2(bf_lo(hist[i].x), bf_hi(hist[i].x));
            x[1] = f2(bf_lo(hist[i].y), bf_hi(hist[i].y));
            x[2] = f2(bf_lo(hist[i].z), bf_hi(hist[i].z));
            x[3] = f2(bf_lo(hist[i].w), bf_hi(hist[i].w));
          }
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) acc[pp] = f2_fma(wt[i][pp], x[pp], acc[pp]);
        }
      }
      uint4 y;
      float lo2, hi2;
      f2_split(acc[0], lo2, hi2); y.x = pack2(lo2, hi2);
      f2_split(acc[1], lo2, hi2); y.y = pack2(lo2, hi2);
      f2_split(acc[2], lo2, hi2); y.z = pack2(lo2, hi2);
      f2_split(acc[3], lo2, hi2); y.w = pack2(lo2, hi2);
      *reinterpret_cast<uint4*>(a.out + t * C + c) = y;
    }

    if (a.state_out == nullptr || W == 0) continue;
    // new state of the requests ending in this chunk: their last W virtual rows
    const int ending = sm.counts[1];
    for (int qq = warp; qq < ending * W; qq += kWarps) {
      const int kk = sm.end_k[qq / W];
      const int jj = qq % W;
      const int st = sm.req_s[kk];
      const int r = sm.req_r[kk];
      const int sj = sm.req_e[kk] - W + jj;  // relative to the chunk start
      uint4 u = make_uint4(0, 0, 0, 0);
      if (sj >= st) {
        int rr = row0 + sj;  // sj in [-W, CH): one wrap either way
        rr = rr < 0 ? rr + NW : wrap(rr);
        const float4 x0 = ring[(rr * 2) * 32 + lane];
        const float4 x1 = ring[(rr * 2 + 1) * 32 + lane];
        u = make_uint4(pack2(x0.x, x0.y), pack2(x0.z, x0.w), pack2(x1.x, x1.y), pack2(x1.z, x1.w));
      } else if (a.state != nullptr) {
        u = ldg16(a.state + (static_cast<int64_t>(r) * W + (W + sj - st)) * C + c);
      }
      *reinterpret_cast<uint4*>(a.state_out + (static_cast<int64_t>(r) * W + jj) * C + c) = u;
    }
  }
  // never leave with a bulk copy in flight into this CTA's shared memory
  // (chunks q .. q+2 may still be in flight only after a timeout above)
  if (tid == 0)
    for (int j = q; j <= nq && j < q + kCsSlots; ++j)
      mbar_wait(smem_u32(bars + j % kCsSlots), static_cast<uint32_t>((j / kCsSlots) & 1), nullptr);
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
  if (T > 0x7fffffff - 2 * kMaxHalo)
    return fail(PLE_ERR_UNSUPPORTED, "%s: %lld tokens is too many", name, static_cast<long long>(T));
  if (!w || (T > 0 && !qsl)) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(w)) return fail(PLE_ERR_INVALID_ARG, "%s: conv taps must be 16-byte aligned", name);
  const size_t state_bytes = static_cast<size_t>(num_reqs) * (K - 1) * dil * C * 2;
  if (state && state_out && state_bytes > 0 && overlaps(state, state_bytes, state_out, state_bytes))
    return fail(PLE_ERR_INVALID_ARG, "%s: conv_state_out overlaps conv_state", name);
  if ((state && !aligned16(state)) || (state_out && !aligned16(state_out)))
    return fail(PLE_ERR_INVALID_ARG, "%s: state buffers must be 16-byte aligned", name);
  return PLE_OK;
}

// Tile of the tiled conv and how its window is staged. A step small enough
// that a tile of 16..112 tokens puts every CTA on the GPU at once takes the
// smallest such tile (one wave: at 256 x 4 decode, 37-token tiles in 448
// CTAs run the conv in 18.3 us against 22.7 us for 16-token tiles in 1024
// CTAs) with per-lane staging (12.5 us against 12.8 us with the TMA copy).
// Otherwise, where the window is one TMA box inside the source tensor, the
// TMA copy with 88-token tiles at 4 CTAs per SM (88.6 us at 32k tokens and
// 28.7 us at 8k against 101.8 and 30.1 us for per-lane staging with
// 112-token tiles at 3 per SM; 112-token TMA tiles at 3 per SM 89.8 and
// 29.5 us); else per-lane staging with 112 tokens when that still gives ~4
// CTAs per SM (each CTA's fixed cost -- request search, one load round
// trip, two barriers -- spread over more tokens: 30.9 us at 8k prefill
// against 32.3 us for 64 and 33.6 us for 128), else 64, halved until ~4 CTAs
// per SM. Measured on a GB300. PLE_CONV_TILE overrides the tile and
// PLE_CONV_TMA = 0 | 1 the staging (launch-shape sweeps and tests).
struct ConvTile {
  int tile;
  bool tma;
};

ConvTile conv_tile(int64_t T, int C, int K, int W, int64_t src_cols) {
  const int64_t slices = (C + kConvSlice - 1) / kConvSlice;
  const int64_t want = 4 * static_cast<int64_t>(num_sms());
  auto ctas = [&](int tile) { return ((T + tile - 1) / tile) * slices; };
  auto tma_fits = [&](int tile) {
    return src_cols >= kConvSlice && T >= tile + W && tile + W <= 256;
  };
  // CTAs per SM of per-lane staging: the register cap of the kernel (3 for
  // K <= 4, else 2), or fewer when the shared memory of a 112-token tile
  // does not fit
  const int64_t by_smem = static_cast<int64_t>(smem_per_sm()) /
                          static_cast<int64_t>(conv_smem_bytes(112, W) + 1024);
  const int64_t per_sm = by_smem < (K <= 4 ? 3 : 2) ? by_smem : (K <= 4 ? 3 : 2);
  const int64_t per_slice = per_sm * num_sms() / slices;  // tiles of one slice in one wave
  ConvTile t{0, false};
  if (per_slice >= 1) {
    const int64_t one_wave = (T + per_slice - 1) / per_slice;
    if (one_wave >= 16 && one_wave <= 112) t.tile = static_cast<int>(one_wave);
  }
  if (t.tile == 0) {
    if (K <= 4 && tma_fits(88)) {
      t = {88, true};
    } else if (tma_fits(112)) {
      t = {112, true};
    } else {
      t.tile = 112;
      if (ctas(t.tile) < want) {
        t.tile = 64;
        while (t.tile > 8 && ctas(t.tile) < want) t.tile >>= 1;
      }
    }
  }
  if (const char* e = getenv("PLE_CONV_TILE")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 128) t.tile = v;
  }
  if (const char* e = getenv("PLE_CONV_TMA")) t.tma = atoi(e) != 0;
  if (t.tma && !tma_fits(t.tile)) t.tma = false;
  return t;
}

template <bool GATED>
ple_status launch_conv(const ConvArgs& a, const float* g, cudaStream_t stream, const char* name) {
  const int W = (a.K - 1) * a.dil;
  const int slices = (a.C + kConvSlice - 1) / kConvSlice;
  // Tiled kernel by default (measured faster at 8k prefill and 256 x 4
  // decode); PLE_CONV_MODE=stream selects the streaming kernel (comparison
  // sweeps and tests: both give the same bits).
  const char* mode = getenv("PLE_CONV_MODE");
  const bool tiled = !(mode != nullptr && strcmp(mode, "stream") == 0);
  int param = 0;
  size_t smem = 0;
  dim3 grid;
  // The tiled kernel's window is one TMA copy (conv_tile: where the box of
  // 256 columns x tile + W rows lies inside the source tensor, kv's value
  // half for the gated pass, x otherwise) or per-lane loads.
  bool use_tma = false;
  const int64_t cols = GATED ? 2 * static_cast<int64_t>(a.C) : a.C;
  if (tiled) {
    const ConvTile ct = conv_tile(a.T, a.C, a.K, W, cols);
    param = ct.tile;
    use_tma = ct.tma;
    smem = conv_smem_bytes(ct.tile, W);
    grid = dim3(static_cast<unsigned>((a.T + ct.tile - 1) / ct.tile), static_cast<unsigned>(slices));
  } else {
    const int CH = conv_stream_chunk(W);
    param = CH;
    smem = conv_stream_smem(CH, W);
    // about two CTAs per SM, each over a contiguous token range of one slice
    int64_t ranges = (2 * static_cast<int64_t>(num_sms()) + slices - 1) / slices;
    const int64_t max_ranges = (a.T + 15) / 16;
    if (ranges > max_ranges) ranges = max_ranges;
    if (ranges < 1) ranges = 1;
    if (const char* e = getenv("PLE_CONV_RANGES")) {
      const long v = atol(e);
      if (v >= 1 && v <= 65535) ranges = v;
    }
    grid = dim3(static_cast<unsigned>(ranges), static_cast<unsigned>(slices));
  }
  using TiledFn = void (*)(ConvArgs, const float*, int, CUtensorMap, int);
  using StreamFn = void (*)(ConvArgs, const float*, int);
  TiledFn tiled_fn = nullptr;
  StreamFn stream_fn = nullptr;
#define PLE_CONV_CASE(KK)                                                                    \
  case KK:                                                                                   \
    tiled_fn = use_tma ? conv_kernel<GATED, KK, true> : conv_kernel<GATED, KK, false>;      \
    stream_fn = conv_stream_kernel<GATED, KK>;                                               \
    break;
  switch (a.K) {
    PLE_CONV_CASE(1)
    PLE_CONV_CASE(2)
    PLE_CONV_CASE(3)
    PLE_CONV_CASE(4)
    PLE_CONV_CASE(5)
    PLE_CONV_CASE(6)
    PLE_CONV_CASE(7)
    default:
    PLE_CONV_CASE(8)
  }
#undef PLE_CONV_CASE
  const void* kernel = tiled ? reinterpret_cast<const void*>(tiled_fn)
                             : reinterpret_cast<const void*>(stream_fn);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return check_cuda(err, name);
  if (tiled) {
    CUtensorMap map{};
    int tma_col0 = -1;
    if (use_tma) {
      const int rows = param + W;
      auto encode = tensor_map_encoder();
      if (encode == nullptr) return fail(PLE_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", name);
      cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(a.T)};
      cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
      cuuint32_t box[2] = {static_cast<cuuint32_t>(kConvSlice), static_cast<cuuint32_t>(rows)};
      cuuint32_t elem_strides[2] = {1, 1};
      CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<ple_bf16_t*>(a.src), dims, strides, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(PLE_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", name,
                    static_cast<int>(r));
      tma_col0 = GATED ? a.C : 0;
    }
    err = launch_kernel(tiled_fn, grid, dim3(kConvThreads), smem, stream, 1, a, g, param, map,
                        tma_col0);
  } else {
    err = launch_kernel(stream_fn, grid, dim3(kConvThreads), smem, stream, 1, a, g, param);
  }
  if (err != cudaSuccess) return check_cuda(err, name);
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
  if (hidden_size > kMaxGateC)
    return fail(PLE_ERR_UNSUPPORTED, "ple_gate: hidden_size %d above %d", hidden_size, kMaxGateC);
  if (num_tokens == 0) return PLE_OK;
  if (!hidden || !kv || !gamma_h || !gamma_k || !out)
    return fail(PLE_ERR_INVALID_ARG, "ple_gate: null pointer");
  if (!aligned16(hidden) || !aligned16(kv) || !aligned16(gamma_h) || !aligned16(gamma_k) ||
      !aligned16(out))
    return fail(PLE_ERR_INVALID_ARG, "ple_gate: buffers must be 16-byte aligned");
  return gate_pass<true>(hidden, kv, gamma_h, gamma_k, eps, num_tokens, hidden_size, out,
                         gate_out, nullptr, stream, "ple_gate");
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
  if (gated && C > kMaxGateC)
    return fail(PLE_ERR_UNSUPPORTED, "%s: hidden_size %d above %d", name, C, kMaxGateC);
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
  a.src = src;
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
  a.dev_err = dev_err;
  if (!gated) return launch_conv<false>(a, nullptr, stream, name);
  s = gate_pass<false>(hidden, src, gamma_h, gamma_k, eps, T, C, nullptr, gate_out, dev_err,
                       stream, name);
  if (s != PLE_OK) return s;
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

PLE_EXPORT ple_status ple_gated_conv(const ple_bf16_t* kv, const float* gate,
                                     const int32_t* query_start_loc, int32_t num_reqs,
                                     int64_t num_tokens, int32_t hidden_size,
                                     const ple_bf16_t* w, int32_t kernel_size, int32_t dilation,
                                     const ple_bf16_t* conv_state, ple_bf16_t* conv_state_out,
                                     ple_bf16_t* out, int32_t* dev_err, cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_gated_conv";
  ple_status s = validate_conv(query_start_loc, num_reqs, num_tokens, hidden_size, w, kernel_size,
                               dilation, conv_state, conv_state_out, name);
  if (s != PLE_OK) return s;
  const size_t state_bytes =
      static_cast<size_t>(num_reqs) * (kernel_size - 1) * dilation * hidden_size * 2;
  if (num_tokens == 0) return copy_carry(conv_state_out, conv_state, state_bytes, stream);
  if (!kv || !gate || !out) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(kv) || !aligned16(out))
    return fail(PLE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", name);
  ConvArgs a{};
  a.src = kv;
  a.qsl = query_start_loc;
  a.num_reqs = num_reqs;
  a.T = num_tokens;
  a.C = hidden_size;
  a.w = w;
  a.K = kernel_size;
  a.dil = dilation;
  a.state = conv_state;
  a.state_out = conv_state_out;
  a.out = out;
  a.dev_err = dev_err;
  return launch_conv<true>(a, gate, stream, name);
}
