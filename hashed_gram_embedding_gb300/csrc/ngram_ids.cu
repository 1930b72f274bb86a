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
// are contiguous. Each thread searches query_start_loc for its token's
// request (cached loads); the heads' constants are staged in shared memory;
// the hash itself is ngram_id (ngram_hash.cuh).
#include "ngram_hash.cuh"

namespace ple {
namespace {

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

  // The heads' constants are staged in shared memory (lanes index different
  // heads); every thread then finds its token's request itself with a
  // binary search of query_start_loc (a few dependent loads that hit L1:
  // the whole array is a few hundred bytes), so the block waits at one
  // barrier only.
  __shared__ NgramHeadsSmem hs;
  stage_ngram_heads(k, num_heads, hs);
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  check_qsl(qsl, num_reqs, num_tokens, i, dev_err);

  // Carry-over: last ctx_len tokens of each request's virtual sequence.
  if (ctx_out != nullptr && i < static_cast<uint32_t>(num_reqs) * static_cast<uint32_t>(ctx_len))
    ngram_carry(input_ids, num_tokens, qsl, num_reqs, ctx, ctx_len, eos, i, ctx_out);

  if (i >= work) return;
  const uint32_t t32 = i / static_cast<uint32_t>(num_heads);
  const int h = static_cast<int>(i - t32 * static_cast<uint32_t>(num_heads));
  const int64_t t = t32;

  // Last request whose start is <= t (the right-sided search of the pages'
  // CPU branch, clamped).
  const int r = find_request(qsl, num_reqs, t);
  const int64_t start = __ldg(qsl + r);
  const int64_t pos = t - start;  // position inside the request

  out[i] = ngram_id(input_ids, ctx, ctx_len, eos, t, pos, r, h, heads_per_ngram, k, hs);
}

}  // namespace

ple_status make_ngram_consts(int32_t ctx_len, int32_t heads_per_ngram,
                             const int64_t* layer_multipliers, const int64_t* vocab_sizes,
                             const int64_t* offsets, NgramConsts* k, int* num_heads,
                             const char* name) {
  if (ctx_len < 1 || ctx_len > PLE_MAX_CTX_LEN)
    return fail(PLE_ERR_INVALID_ARG, "%s: ctx_len %d not in [1, %d]", name, ctx_len,
                PLE_MAX_CTX_LEN);
  if (heads_per_ngram < 1)
    return fail(PLE_ERR_INVALID_ARG, "%s: heads_per_ngram must be >= 1 "
                "(empty head shards are rejected)", name);
  const int H = ctx_len * heads_per_ngram;
  if (H > PLE_MAX_HEADS)
    return fail(PLE_ERR_INVALID_ARG, "%s: %d heads > %d", name, H, PLE_MAX_HEADS);
  if (!layer_multipliers || !vocab_sizes || !offsets)
    return fail(PLE_ERR_INVALID_ARG, "%s: null host constant array", name);
  *k = NgramConsts{};
  for (int s = 0; s <= ctx_len; ++s) k->mult[s] = layer_multipliers[s];
  for (int h = 0; h < H; ++h) {
    const int64_t V = vocab_sizes[h];
    if (V < 1)
      return fail(PLE_ERR_INVALID_ARG, "%s: vocab_sizes[%d] = %lld < 1", name, h,
                  static_cast<long long>(V));
    k->vocab[h] = V;
    k->offset[h] = offsets[h];
    const unsigned __int128 two64 = static_cast<unsigned __int128>(1) << 64;
    k->magic[h] = (V == 1) ? 0 : static_cast<uint64_t>(two64 / static_cast<uint64_t>(V));
    k->pow64_mod[h] = static_cast<uint64_t>(two64 % static_cast<uint64_t>(V));
  }
  *num_heads = H;
  return PLE_OK;
}

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
  NgramConsts k{};
  int num_heads = 0;
  ple_status cs = make_ngram_consts(ctx_len, heads_per_ngram, layer_multipliers, vocab_sizes,
                                    offsets, &k, &num_heads, "ple_ngram_ids");
  if (cs != PLE_OK) return cs;
  if (num_reqs < 0 || (num_reqs == 0 && num_tokens > 0))
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: num_reqs must be >= 1 when there are tokens");
  if (ngram_context_out && ngram_context &&
      overlaps(ngram_context, sizeof(int32_t) * num_reqs * ctx_len, ngram_context_out,
               sizeof(int32_t) * num_reqs * ctx_len))
    return fail(PLE_ERR_INVALID_ARG, "ple_ngram_ids: ngram_context_out overlaps ngram_context");

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
