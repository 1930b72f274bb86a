// The n-gram hash of one (token, head), shared by ple_ngram_ids and the fused
// ple_ngram_lookup.
//
// Source: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), 关键源码片段:
// compute_ngram_ids and the _ple_ngram_ids_kernel skeleton -- prefix tokens
// from the request or from ngram_context (EOS before a request's history),
// EOS crossing, XOR mix of token * multiplier, per-head reduction into the
// head's table partition with torch.remainder (floor-mod) int64 semantics.
//
// The floor-mod uses a multiply-high instead of a 64-bit division:
//   magic = floor(2^64 / V)  =>  q = umulhi(u, magic) is floor(u / V) or one
//   less, so r = u - q*V lies in [0, 2V) and one conditional subtraction gives
//   u mod V. A negative int64 m is u - 2^64, so floor_mod(m, V) is
//   (u mod V - 2^64 mod V) mod V.
// The constants (multipliers, V, O, magic numbers) travel by value in the
// kernel's parameter block: no device allocation, graph-capture friendly.
#pragma once

#include "common.cuh"

namespace ple {

constexpr int kStagedBounds = 4096;  // query_start_loc entries staged in shared memory

struct NgramConsts {
  int64_t mult[PLE_MAX_CTX_LEN + 1];
  int64_t vocab[PLE_MAX_HEADS];
  int64_t offset[PLE_MAX_HEADS];
  uint64_t magic[PLE_MAX_HEADS];     // floor(2^64 / V), 0 when V == 1
  uint64_t pow64_mod[PLE_MAX_HEADS]; // 2^64 mod V
};

// Host: check the hash arguments and fill the constants; *num_heads =
// ctx_len * heads_per_ngram. Errors name `name`.
ple_status make_ngram_consts(int32_t ctx_len, int32_t heads_per_ngram,
                             const int64_t* layer_multipliers, const int64_t* vocab_sizes,
                             const int64_t* offsets, NgramConsts* k, int* num_heads,
                             const char* name);

// Per-head constants staged in shared memory: the lanes of a warp index
// different heads, and a lane-varying index into the parameter block would
// serialise on the constant cache.
struct NgramHeadsSmem {
  uint64_t vocab[PLE_MAX_HEADS], offset[PLE_MAX_HEADS];
  uint64_t magic[PLE_MAX_HEADS], pow64[PLE_MAX_HEADS];
};

__device__ __forceinline__ void stage_ngram_heads(const NgramConsts& k, int num_heads,
                                                  NgramHeadsSmem& hs) {
  for (int h = threadIdx.x; h < num_heads; h += blockDim.x) {
    hs.vocab[h] = static_cast<uint64_t>(k.vocab[h]);
    hs.offset[h] = static_cast<uint64_t>(k.offset[h]);
    hs.magic[h] = k.magic[h];
    hs.pow64[h] = k.pow64_mod[h];
  }
}

__device__ __forceinline__ int64_t floor_mod(int64_t m, uint64_t V,
                                             uint64_t magic, uint64_t pow64_mod) {
  if (V == 1) return 0;
  const uint64_t u = static_cast<uint64_t>(m);
  uint64_t r = u - __umul64hi(u, magic) * V;
  if (r >= V) r -= V;
  if (m < 0) r = (r >= pow64_mod) ? r - pow64_mod : r + V - pow64_mod;
  return static_cast<int64_t>(r);
}

// id of head h for token t at position pos of request r (pos = t - start):
// tokens at lags 1 .. n-1 come from the request, before its start from
// ngram_context[r] (oldest first; NULL = EOS); an EOS at lag j >= 1 turns
// every larger lag into EOS; XOR of the wrapped products token * mult[lag];
// floor-mod into the head's partition plus its offset.
__device__ __forceinline__ int64_t ngram_id(const int32_t* __restrict__ input_ids,
                                            const int32_t* __restrict__ ctx, int ctx_len,
                                            int eos, int64_t t, int64_t pos, int r, int h,
                                            int heads_per_ngram, const NgramConsts& k,
                                            const NgramHeadsSmem& hs) {
  const int order_lags = h / heads_per_ngram + 1;  // n - 1 for this head
  int64_t mixed = 0;
  bool crossed = false;
  for (int s = 0; s <= order_lags; ++s) {
    int32_t x;
    const int64_t q = pos - s;
    if (q >= 0) {
      x = (t - s >= 0) ? __ldg(input_ids + (t - s)) : eos;
    } else {
      const int64_t hist = ctx_len + q;  // history slot, oldest first
      x = (ctx != nullptr && hist >= 0)
              ? __ldg(ctx + static_cast<int64_t>(r) * ctx_len + hist) : eos;
    }
    if (s >= 1) {
      if (crossed) x = eos;
      else if (x == eos) crossed = true;
    }
    const uint64_t term = static_cast<uint64_t>(static_cast<int64_t>(x)) *
                          static_cast<uint64_t>(k.mult[s]);
    mixed = (s == 0) ? static_cast<int64_t>(term)
                     : static_cast<int64_t>(static_cast<uint64_t>(mixed) ^ term);
  }
  return floor_mod(mixed, hs.vocab[h], hs.magic[h], hs.pow64[h]) +
         static_cast<int64_t>(hs.offset[h]);
}

// Carry-over entry i of ngram_context_out ([num_reqs][ctx_len]): the last
// ctx_len tokens of request r's virtual sequence history ++ segment.
__device__ __forceinline__ void ngram_carry(const int32_t* __restrict__ input_ids,
                                            int64_t num_tokens, const int32_t* __restrict__ qsl,
                                            int num_reqs, const int32_t* __restrict__ ctx,
                                            int ctx_len, int eos, int64_t i,
                                            int32_t* __restrict__ ctx_out) {
  const int r = static_cast<int>(i / ctx_len);
  const int j = static_cast<int>(i - static_cast<int64_t>(r) * ctx_len);
  int64_t start, end;
  request_span(qsl, num_reqs, num_tokens, r, &start, &end);
  const int64_t p = (end - start) + j;  // index into history ++ segment
  int32_t v;
  if (p < ctx_len) v = ctx ? __ldg(ctx + static_cast<int64_t>(r) * ctx_len + p) : eos;
  else v = __ldg(input_ids + start + (p - ctx_len));
  ctx_out[i] = v;
}

}  // namespace ple
