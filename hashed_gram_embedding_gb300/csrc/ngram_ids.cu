// ple_ngram_ids: ragged n-gram hash ids.
//
// Source: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), section 关键源码片段:
// compute_ngram_ids (request of a token = right-sided search of
// query_start_loc minus one, clamped; EOS padding before a request's first
// token) and the _ple_ngram_ids_kernel skeleton (prefix tokens from the
// request or from ngram_context; EOS crossing; XOR mix of token*multiplier;
// per-head reduction into the head's table partition; torch.remainder int64
// semantics).
//
// Design: one thread per (token, head) output, so the int64 stores of a warp
// are contiguous. Each thread binary-searches its request in query_start_loc
// (L1-resident), reads at most NGRAM_CONTEXT_LEN + 1 tokens, and reduces with
// a multiply-high floor-mod instead of a 64-bit division:
//   magic = floor(2^64 / V)  =>  q = umulhi(u, magic) is floor(u / V) or one
//   less, so r = u - q*V lies in [0, 2V) and one conditional subtraction gives
//   u mod V. A negative int64 m is u - 2^64, so floor_mod(m, V) is
//   (u mod V - 2^64 mod V) mod V.
// The constants (multipliers, V, O, magic numbers) travel by value in the
// kernel's parameter block: no device allocation, graph-capture friendly.
#include "common.cuh"

namespace ple {
namespace {

constexpr int kStagedBounds = 4096;  // query_start_loc entries staged in shared memory

struct NgramConsts {
  int64_t mult[PLE_MAX_CTX_LEN + 1];
  int64_t vocab[PLE_MAX_HEADS];
  int64_t offset[PLE_MAX_HEADS];
  uint64_t magic[PLE_MAX_HEADS];     // floor(2^64 / V), 0 when V == 1
  uint64_t pow64_mod[PLE_MAX_HEADS]; // 2^64 mod V
};

__device__ __forceinline__ int64_t floor_mod(int64_t m, uint64_t V,
                                             uint64_t magic, uint64_t pow64_mod) {
  if (V == 1) return 0;
  const uint64_t u = static_cast<uint64_t>(m);
  uint64_t r = u - __umul64hi(u, magic) * V;
  if (r >= V) r -= V;
  if (m < 0) r = (r >= pow64_mod) ? r - pow64_mod : r + V - pow64_mod;
  return static_cast<int64_t>(r);
}

__global__ void __launch_bounds__(256)
ngram_ids_kernel(const int32_t* __restrict__ input_ids, int64_t num_tokens,
                 const int32_t* __restrict__ qsl, int num_reqs,
                 const int32_t* __restrict__ ctx, int ctx_len, int eos,
                 int heads_per_ngram, int num_heads,
                 int64_t* __restrict__ out, int32_t* __restrict__ ctx_out,
                 int32_t* dev_err, const __grid_constant__ NgramConsts k) {
  // 32-bit indices: the host caps num_tokens * num_heads below 2^31.
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t work = static_cast<uint32_t>(num_tokens) * static_cast<uint32_t>(num_heads);

  // Request boundaries staged once per block (one coalesced load); the
  // block's first token is searched once, every thread then steps forward
  // from there (a block spans 256 / num_heads consecutive tokens).
  __shared__ int32_t qsl_s[kStagedBounds];
  __shared__ int r_first_s;
  // Per-head constants: the lanes of a warp index different heads, so they
  // are read from shared memory (a lane-varying index into the parameter
  // block would serialise on the constant cache).
  __shared__ uint64_t vocab_s[PLE_MAX_HEADS], offset_s[PLE_MAX_HEADS];
  __shared__ uint64_t magic_s[PLE_MAX_HEADS], pow64_s[PLE_MAX_HEADS];
  const bool staged = num_reqs < kStagedBounds;
  for (int h = threadIdx.x; h < num_heads; h += blockDim.x) {
    vocab_s[h] = static_cast<uint64_t>(k.vocab[h]);
    offset_s[h] = static_cast<uint64_t>(k.offset[h]);
    magic_s[h] = k.magic[h];
    pow64_s[h] = k.pow64_mod[h];
  }
  pdl_wait();
  pdl_trigger();
  if (staged)
    for (int r = threadIdx.x; r <= num_reqs; r += blockDim.x) qsl_s[r] = __ldg(qsl + r);
  __syncthreads();
  const uint32_t i_first = blockIdx.x * blockDim.x;
  if (threadIdx.x == 0 && i_first < work) {
    const int64_t t_first = i_first / static_cast<uint32_t>(num_heads);
    int r;
    if (staged) {
      int lo = 0, hi = num_reqs + 1;  // count of boundaries <= t_first
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(qsl_s[mid]) <= t_first) lo = mid + 1; else hi = mid;
      }
      r = lo - 1 < 0 ? 0 : (lo - 1 >= num_reqs ? num_reqs - 1 : lo - 1);
    } else {
      r = find_request(qsl, num_reqs, t_first);
    }
    r_first_s = r;
  }
  __syncthreads();

  check_qsl(qsl, num_reqs, num_tokens, i, dev_err);

  // Carry-over: last ctx_len tokens of each request's virtual sequence.
  if (ctx_out != nullptr && i < static_cast<uint32_t>(num_reqs) * static_cast<uint32_t>(ctx_len)) {
    const int r = static_cast<int>(i / static_cast<uint32_t>(ctx_len));
    const int j = static_cast<int>(i - static_cast<uint32_t>(r) * ctx_len);
    int64_t start, end;
    request_span(qsl, num_reqs, num_tokens, r, &start, &end);
    const int64_t len = end - start;
    const int64_t p = len + j;  // index into history ++ segment
    int32_t v;
    if (p < ctx_len) v = ctx ? __ldg(ctx + static_cast<int64_t>(r) * ctx_len + p) : eos;
    else v = __ldg(input_ids + start + (p - ctx_len));
    ctx_out[i] = v;
  }

  if (i >= work) return;
  const uint32_t t32 = i / static_cast<uint32_t>(num_heads);
  const int h = static_cast<int>(i - t32 * static_cast<uint32_t>(num_heads));
  const int64_t t = t32;
  const int order_lags = h / heads_per_ngram + 1;  // n - 1 for this head

  // Last request whose start is <= t (the right-sided search of the pages'
  // CPU branch, clamped): step forward from the block's first request.
  int r = r_first_s;
  int64_t start;
  if (staged) {
    while (r + 1 < num_reqs && static_cast<int64_t>(qsl_s[r + 1]) <= t) ++r;
    start = qsl_s[r];
  } else {
    r = find_request(qsl, num_reqs, t);
    start = __ldg(qsl + r);
  }
  const int64_t pos = t - start;  // position inside the request

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
  out[i] = floor_mod(mixed, vocab_s[h], magic_s[h], pow64_s[h]) +
           static_cast<int64_t>(offset_s[h]);
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_ngram_ids(const int32_t* input_ids, int64_t num_tokens,
                                    const int32_t* query_start_loc, int32_t num_reqs,
                                    const int32_t* ngram_context, int32_t ctx_len,
                                    const int64_t* layer_multipliers,
                                    const int64_t* vocab_sizes, const int64_t* offsets,
                                    int32_t eos_token_id, int32_t heads_per_ngram,
                                    int64_t* out, int32_t* ngram_context_out,
                                    int32_t* dev_err, cudaStream_t stream) {
  using namespace ple;
  if (num_tokens < 0) return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: num_tokens < 0");
  if (ctx_len < 1 || ctx_len > PLE_MAX_CTX_LEN)
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: ctx_len %d not in [1, %d]", ctx_len,
                PLE_MAX_CTX_LEN);
  if (heads_per_ngram < 1)
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: heads_per_ngram must be >= 1 "
                "(empty head shards are rejected)");
  const int num_heads = ctx_len * heads_per_ngram;
  if (num_heads > PLE_MAX_HEADS)
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: %d heads > %d", num_heads, PLE_MAX_HEADS);
  if (num_reqs < 0 || (num_reqs == 0 && num_tokens > 0))
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: num_reqs must be >= 1 when there are tokens");
  if (!layer_multipliers || !vocab_sizes || !offsets)
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: null host constant array");
  if (ngram_context_out && ngram_context &&
      overlaps(ngram_context, sizeof(int32_t) * num_reqs * ctx_len, ngram_context_out,
               sizeof(int32_t) * num_reqs * ctx_len))
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: ngram_context_out overlaps ngram_context");

  NgramConsts k{};
  for (int s = 0; s <= ctx_len; ++s) k.mult[s] = layer_multipliers[s];
  for (int h = 0; h < num_heads; ++h) {
    const int64_t V = vocab_sizes[h];
    if (V < 1) return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: vocab_sizes[%d] = %lld < 1",
                           h, static_cast<long long>(V));
    k.vocab[h] = V;
    k.offset[h] = offsets[h];
    const unsigned __int128 two64 = static_cast<unsigned __int128>(1) << 64;
    k.magic[h] = (V == 1) ? 0 : static_cast<uint64_t>(two64 / static_cast<uint64_t>(V));
    k.pow64_mod[h] = static_cast<uint64_t>(two64 % static_cast<uint64_t>(V));
  }

  if (num_tokens == 0) {
    // Zero tokens: nothing to hash; the carry-over is the history itself.
    if (ngram_context_out == nullptr || num_reqs == 0) return PLE_OK;
    if (ngram_context != nullptr)
      return copy_carry(ngram_context_out, ngram_context,
                        sizeof(int32_t) * num_reqs * ctx_len, stream);
    // No history means ctx_len EOS tokens: the kernel below writes them.
  }
  if ((num_tokens > 0 && (!input_ids || !out)) || !query_start_loc)
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: null device pointer");

  const int64_t work = num_tokens * num_heads;
  const int64_t carry = static_cast<int64_t>(num_reqs) * ctx_len;
  const int64_t threads = work > carry ? work : carry;
  const int64_t blocks = (threads + 255) / 256;
  if (threads >= (int64_t(1) << 31))
    return fail(PLE_ERR_UNSUPPORTED, "ple_ngram_ids: num_tokens * heads must stay below 2^31");
  cudaError_t lerr = launch_kernel(ngram_ids_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                   stream, 1, input_ids, num_tokens, query_start_loc, num_reqs,
                                   ngram_context, ctx_len, eos_token_id, heads_per_ngram,
                                   num_heads, out, ngram_context_out, dev_err, k);
  if (lerr != cudaSuccess) return check_cuda(lerr, "ple_ngram_ids launch");
  return check_cuda(cudaGetLastError(), "ple_ngram_ids launch");
}
