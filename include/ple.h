/*
 * ple.h -- C ABI of libple: the per-layer n-gram embedding (PLE / Engram)
 * lookup path for one GB300 (sm_103a) GPU.
 *
 * The path (one transformer layer):
 *   ple_ngram_ids  ragged n-gram hash ids        -> ids [T][H] int64
 *   ple_lookup     multi-head row gather         -> emb [T][H*D] bf16
 *                  (ple_ngram_lookup: both in one kernel)
 *   ple_kv_proj    merged key/value projection   -> kv  [T][2C] bf16
 *   ple_gate_conv  RMSNorm + sigmoid gate, then the dilated causal depthwise
 *                  short conv                    -> y   [T][C] bf16
 * with ple_gate / ple_conv as the two halves of ple_gate_conv, and
 * ple_lookup_prefetch / ple_wait for a gather on a side stream (a table in
 * pinned host memory read over UVA, overlapped with other work). The same
 * layer with the gate's reductions moved into the projection:
 *   ple_kv_proj_gate  projection + gate scalars -> v half of kv, g [T] f32
 *   ple_gated_conv    short conv of u = g * v   -> y   [T][C] bf16
 *
 * Sources (page titles abbreviated):
 *   PR#54517 report "[Qwen3.8-Flash-Next] Fuse Qwen4Exp PLE kernels":
 *     section 关键源码片段 (compute_ngram_ids and its CPU branch; the
 *     _ple_ngram_ids_kernel signature and skeleton), 实现拆解 items 1, 2, 4
 *     (merged kv_proj; ple_ngram_ids / ple_gate / ple_conv; short-conv state).
 *   PR#54371 report "[Qwen4Exp] Support UVA PLE-offload and Engram tensor
 *     parallelism": 实现拆解 items 1 and 4, 关键源码片段 (device and
 *     pinned-host embedding backends, start_prefetch, BF16/FP8 weights).
 *   PR#56512 report "[DS V4.1][Engram] Support async prefetch ...":
 *     功能与动机 and 实现拆解 item 4 (side-stream prefetch with a reduced grid,
 *     the consumer waiting on the side stream), 关键源码片段 (pinned check).
 *
 * Conventions for every entry point:
 *   - Buffers are caller-owned. Unless a comment says "host", a pointer is
 *     device memory (or any memory the GPU can address, e.g. managed).
 *     The one exception is the table of ple_lookup in PLE_HOST_UVA mode,
 *     which must be pinned (cudaHostAlloc) or registered (cudaHostRegister)
 *     host memory.
 *   - Calls are asynchronous on the given stream (0 = legacy default stream)
 *     and never synchronise it, except ple_wait with a host timeout.
 *   - The library allocates no device or host memory (except the explicit
 *     ple_host_table_alloc, and the graph and event objects of the step
 *     runtime, which the caller destroys) and keeps no state between calls
 *     other than the thread-local error text.
 *   - bf16 data is passed as 16-bit containers (ple_bf16_t): IEEE binary32
 *     truncated to its high half, row-major.
 *   - A call returns PLE_OK when its work was enqueued. Argument errors found
 *     on the host return PLE_ERR_INVALID_ARG / PLE_ERR_UNSUPPORTED and enqueue
 *     nothing. Errors that only the GPU can see (an id outside the table,
 *     invalid query_start_loc contents, a pipeline wait that gave up) are
 *     OR-ed as PLE_DEVERR_* bits into the optional device word `dev_err`
 *     (pass NULL to ignore them); the kernel then writes zeros for the
 *     affected rows instead of touching memory out of range. The caller
 *     clears *dev_err before the call when it wants a fresh reading.
 *   - num_tokens == 0 is a no-op returning PLE_OK (a zero-token prefetch
 *     returns early, PR#54371 report, start_prefetch); carry-over outputs
 *     (ngram_context_out, conv_state_out) are then copied from their inputs.
 *   - ple_last_error() gives a human-readable reason for the last non-OK
 *     status returned on the calling host thread.
 */
#ifndef PLE_H_
#define PLE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ple_bf16_t;

typedef enum {
  PLE_OK = 0,
  PLE_ERR_INVALID_ARG = 1,  /* bad pointer / size / layout found on the host */
  PLE_ERR_UNSUPPORTED = 2,  /* valid but not handled (e.g. row not 16-byte sized) */
  PLE_ERR_CUDA = 3,         /* a CUDA runtime call failed (text in ple_last_error) */
  PLE_ERR_TIMEOUT = 4,      /* ple_wait gave up before the event completed */
  PLE_ERR_BOUNDS = 5        /* reserved for callers mapping PLE_DEVERR_BOUNDS */
} ple_status;

/* Bits OR-ed into the optional device word `dev_err`. */
#define PLE_DEVERR_BOUNDS 1   /* an id was outside [0, table_rows): row zeroed */
#define PLE_DEVERR_QSL 2      /* query_start_loc not 0-based / non-decreasing / <= T */
#define PLE_DEVERR_TIMEOUT 4  /* a kernel pipeline wait exceeded its limit */

/* Table element types: bf16 rows; fp8 e4m3 rows with a float32 scale per row;
 * fp8 e4m3 rows with one float32 scale for the whole table (the pages'
 * single weight_scale). */
typedef enum { PLE_BF16 = 0, PLE_FP8_E4M3 = 1, PLE_FP8_E4M3_TENSOR = 2 } ple_dtype;
typedef enum { PLE_HBM = 0, PLE_HOST_UVA = 1 } ple_table_loc;
/* How a table is split across the ranks of an exchange group
 * (ple_lookup_shard): by heads, or by contiguous row ranges. */
typedef enum { PLE_SHARD_HEADS = 0, PLE_SHARD_ROWS = 1 } ple_shard_kind;

/* Limits of ple_ngram_ids (constants travel in the kernel's parameter block). */
#define PLE_MAX_CTX_LEN 7     /* NGRAM_CONTEXT_LEN: n-gram orders 2 .. ctx_len + 1 */
#define PLE_MAX_HEADS 64      /* ctx_len * heads_per_ngram */

/*
 * ple_ngram_ids -- ragged n-gram hash ids of every token.
 * (PR#54517 report, 关键源码片段: compute_ngram_ids, _ple_ngram_ids_kernel.)
 *
 * For token t of request r, over r's virtual sequence
 * S = ngram_context[r] ++ input_ids[segment of r] (history oldest first;
 * NULL history = ctx_len EOS tokens, the EOS padding at request starts),
 * with x_s the token s places back (s = 0 current):
 *   - EOS crossing: an EOS at lag j >= 1 is kept, every lag > j becomes EOS;
 *   - mixed_1 = x_0 * m_0 and mixed_{s+1} = mixed_s XOR (x_s * m_s), all in
 *     wrapping int64 arithmetic (tokens are sign-extended int32);
 *   - order n = s + 1 (s = 1 .. ctx_len) emits heads
 *     h = (n - 2) * heads_per_ngram + j, j < heads_per_ngram:
 *     out[t][h] = floor_mod(mixed_n, V_h) + O_h  (torch.remainder semantics).
 * Token t belongs to the last request whose start is <= t, so empty requests
 * own nothing and tokens at or past query_start_loc[num_reqs] continue the
 * last request (padding of a captured graph).
 *
 *   input_ids          [num_tokens] int32, device.
 *   query_start_loc    [num_reqs + 1] int32, device; must be 0 at [0],
 *                      non-decreasing, and <= num_tokens at [num_reqs]
 *                      (checked on the GPU -> PLE_DEVERR_QSL; ids are then
 *                      still written, from clamped positions).
 *   ngram_context      [num_reqs][ctx_len] int32 device, oldest first, or NULL.
 *   ctx_len            1 .. PLE_MAX_CTX_LEN.
 *   layer_multipliers  [ctx_len + 1] int64, HOST (copied at the call).
 *   vocab_sizes        [H] int64 HOST, each >= 1; H = ctx_len * heads_per_ngram
 *                      <= PLE_MAX_HEADS.
 *   offsets            [H] int64 HOST.
 *   out                [num_tokens][H] int64, device.
 *   ngram_context_out  [num_reqs][ctx_len] int32 device or NULL: the last
 *                      ctx_len tokens of each S (carry-over for the next step);
 *                      must not overlap ngram_context (ping-pong two buffers).
 *   dev_err            optional device word (see conventions).
 * Errors: num_reqs < 1 with num_tokens > 0, bad sizes, overlapping
 * context buffers, V_h < 1 -> PLE_ERR_INVALID_ARG.
 */
ple_status ple_ngram_ids(const int32_t* input_ids, int64_t num_tokens,
                         const int32_t* query_start_loc, int32_t num_reqs,
                         const int32_t* ngram_context, int32_t ctx_len,
                         const int64_t* layer_multipliers,
                         const int64_t* vocab_sizes, const int64_t* offsets,
                         int32_t eos_token_id, int32_t heads_per_ngram,
                         int64_t* out, int32_t* ngram_context_out,
                         int32_t* dev_err, cudaStream_t stream);

/*
 * ple_lookup -- multi-head row gather, bf16 or fp8 e4m3 with a per-row or a
 * whole-table scale. (PR#54371 report: device / pinned-host embedding
 * backends, F.embedding; BF16 / FP8 weight methods. PR#53899 page: FP8 table
 * with one weight_scale.)
 *
 *   out[t][h*D + c] = table[ids[t][h]][c]                                 (bf16)
 *   out[t][h*D + c] = bf16_rn(float(e4m3(table[id][c])) * row_scale[id])  (PLE_FP8_E4M3)
 *   out[t][h*D + c] = bf16_rn(float(e4m3(table[id][c])) * row_scale[0])   (PLE_FP8_E4M3_TENSOR)
 *
 *   ids          [num_tokens][num_heads] int64 device (offsets already added).
 *   table        [table_rows][head_dim] (bf16 or uint8 e4m3 codes). In
 *                PLE_HBM mode device memory; in PLE_HOST_UVA mode pinned or
 *                registered host memory (checked with cudaPointerGetAttributes,
 *                else PLE_ERR_INVALID_ARG), read in place over the host link.
 *                16-byte aligned.
 *   row_scale    float32 device: [table_rows] for PLE_FP8_E4M3, [1] for
 *                PLE_FP8_E4M3_TENSOR; NULL for bf16.
 *   out          [num_tokens][num_heads * head_dim] bf16 device, 16-byte aligned.
 *   max_ctas     0 = a full-GPU grid; > 0 caps the grid (e.g. half the SMs
 *                for a side-stream prefetch that overlaps other kernels).
 * A row's byte size (head_dim * element size) must be a multiple of 16
 * (else PLE_ERR_UNSUPPORTED). Ids outside [0, table_rows) give a zero row
 * and PLE_DEVERR_BOUNDS.
 */
ple_status ple_lookup(const int64_t* ids, int64_t num_tokens, int32_t num_heads,
                      const void* table, int64_t table_rows, int32_t head_dim,
                      ple_dtype dtype, const float* row_scale,
                      ple_table_loc loc, ple_bf16_t* out, int32_t max_ctas,
                      int32_t* dev_err, cudaStream_t stream);

/*
 * ple_lookup_prefetch -- ple_lookup enqueued on `side_stream`, after which
 * `done` is recorded on that stream. The consumer later calls ple_wait
 * (or cudaStreamWaitEvent) before reading `out`.
 * (PR#54371 report: start_prefetch on a prefetch stream; PR#56512 report:
 * lookup on a side stream with a reduced grid, embed() waits on it.)
 * `done` is created by the caller (cudaEventCreateWithFlags, timing disabled
 * is fine). The inputs (ids) must be ready on side_stream: record an event
 * on the producer stream and make side_stream wait on it first.
 */
ple_status ple_lookup_prefetch(const int64_t* ids, int64_t num_tokens,
                               int32_t num_heads, const void* table,
                               int64_t table_rows, int32_t head_dim,
                               ple_dtype dtype, const float* row_scale,
                               ple_table_loc loc, ple_bf16_t* out,
                               int32_t max_ctas, int32_t* dev_err,
                               cudaStream_t side_stream, cudaEvent_t done);

/*
 * ple_lookup_ordered -- ple_lookup with the rows read in table order: the
 * (token, head) items are first sorted by the 2 MiB span of the table their
 * row lies in (a counting sort into `workspace`), then gathered in that order,
 * each row written to its own output slot, so `out` is identical to
 * ple_lookup's. For tables in host memory (PLE_HOST_UVA): the GPU's address
 * translation for host memory has limited reach, and random rows over tens of
 * GB miss it on almost every row (a tenth of the link rate on a GB300), while
 * rows read in table order run at the link rate. Same ids/table/out rules and
 * device error word as ple_lookup. (PR#54371 report: the pinned-host backend
 * reads the rows it needs in place; the ordering is this library's.)
 *   workspace        device memory, 256-byte aligned, at least
 *                    ple_lookup_ordered_workspace(...) bytes (else
 *                    PLE_ERR_INVALID_ARG); its contents on entry do not
 *                    matter and are unspecified afterwards. Two calls in
 *                    flight at once must not share one workspace.
 * Four kernel launches and one memset on `stream`.
 */
size_t ple_lookup_ordered_workspace(int64_t num_tokens, int32_t num_heads,
                                    int64_t table_rows, int32_t head_dim,
                                    ple_dtype dtype);
ple_status ple_lookup_ordered(const int64_t* ids, int64_t num_tokens,
                              int32_t num_heads, const void* table,
                              int64_t table_rows, int32_t head_dim,
                              ple_dtype dtype, const float* row_scale,
                              ple_table_loc loc, ple_bf16_t* out,
                              int32_t max_ctas, void* workspace,
                              size_t workspace_bytes, int32_t* dev_err,
                              cudaStream_t stream);

/*
 * ple_lookup_ordered_static -- ple_lookup_ordered with its scratch in a
 * fixed 8 MiB device array inside the library (one per device) instead of a
 * caller workspace. The pages have no counterpart: it exists for callers
 * that may not allocate device memory on their serving path (an engine that
 * carves all device memory into its own pools at start-up, or a C caller
 * without a device allocator); the call itself allocates nothing.
 *   Same arguments, results and device error word as ple_lookup_ordered,
 *   minus the workspace.
 *   Limit: ple_lookup_ordered_workspace(...) of the call must be at most
 *   8 MiB (for 256-byte rows over a 32 GiB table: up to about 1.9 million
 *   (token, head) items), else PLE_ERR_UNSUPPORTED naming the sizes.
 *   Set-up: the first call on a device looks the array's address up
 *   (cudaGetSymbolAddress) and caches it; make that first call before any
 *   stream capture. Nothing in the scratch has to start at zero: each call
 *   clears the counters it uses on `stream` before the kernels.
 *   Races: all calls on one device share the scratch, so two calls in
 *   flight at once (other streams, other host threads) corrupt each other's
 *   walk order; callers must keep such calls ordered.
 */
ple_status ple_lookup_ordered_static(const int64_t* ids, int64_t num_tokens,
                                     int32_t num_heads, const void* table,
                                     int64_t table_rows, int32_t head_dim,
                                     ple_dtype dtype, const float* row_scale,
                                     ple_table_loc loc, ple_bf16_t* out,
                                     int32_t max_ctas, int32_t* dev_err,
                                     cudaStream_t stream);

/*
 * ple_lookup_shard -- one rank's part of a lookup whose table is split over
 * the ranks of an exchange group, on ids already gathered from every
 * replica of the group.
 * (PR#56512 report, 执行摘要 and 实现拆解 3-4: heads sharded over the
 * engram-DP group in TP-major order, hashes padded and all-gathered, each
 * rank looking up its own heads for every gathered token. PR#54371 report,
 * 实现拆解 3 and 关键源码片段 _get_dp_gather_slot / _gather_dp_ids: the table
 * sharded over ETP = TP x DP ranks, rows combined by a parallel reduce, fp8
 * rows reduced as an int8 view.)
 *
 * For token t < num_tokens and head j < num_heads, with the global row
 * g = ids[t][head_begin + j] and the local row l = g - row_base:
 *   PLE_SHARD_HEADS: the rank's table holds the rows of heads
 *     [head_begin, head_begin + num_heads) of the concatenated table, its
 *     row 0 being global row row_base. out[t][j*D + c] is ple_lookup's value
 *     of local row l (bf16 out; fp8 dequantised with the row's or the
 *     table's scale). l outside [0, table_rows) gives a zero row and
 *     PLE_DEVERR_BOUNDS.
 *   PLE_SHARD_ROWS: the rank's table holds global rows
 *     [row_base, row_base + table_rows). out keeps the table's raw bytes:
 *     bf16 rows as stored, fp8 rows as their e4m3 codes with the float32
 *     scale of row l in scale_out[t][j] (the table's one scale for
 *     PLE_FP8_E4M3_TENSOR). l outside the rank's rows is not an error: the
 *     row's bytes and scale are zero, so adding the ranks' outputs as 8-bit
 *     integers (one nonzero contributor per byte) rebuilds every row exactly.
 *
 *   ids        [num_tokens][ids_heads] int64 device; the columns
 *              [head_begin, head_begin + num_heads) are read.
 *   table      [table_rows][head_dim] (bf16, or uint8 e4m3 codes); device
 *              memory (PLE_HBM) or pinned / registered host memory
 *              (PLE_HOST_UVA), 16-byte aligned.
 *   row_scale  float32 device: [table_rows] (PLE_FP8_E4M3), [1]
 *              (PLE_FP8_E4M3_TENSOR), NULL for bf16.
 *   out        16-byte aligned device: PLE_SHARD_HEADS: [num_tokens]
 *              [num_heads * head_dim] bf16; PLE_SHARD_ROWS: the same shape
 *              in the table's element type (bf16 bits or e4m3 codes).
 *   scale_out  [num_tokens][num_heads] float32 device, required for an fp8
 *              table with PLE_SHARD_ROWS; ignored otherwise.
 *   max_ctas   as in ple_lookup.
 * Errors: bad sizes, head range outside [0, ids_heads), unknown dtype /
 * kind / location, a missing scale -> PLE_ERR_INVALID_ARG; a row that is not
 * a multiple of 16 bytes -> PLE_ERR_UNSUPPORTED. num_tokens == 0 is a no-op.
 */
ple_status ple_lookup_shard(const int64_t* ids, int64_t num_tokens, int32_t ids_heads,
                            int32_t head_begin, int32_t num_heads, const void* table,
                            int64_t table_rows, int64_t row_base, int32_t head_dim,
                            ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                            ple_shard_kind kind, void* out, float* scale_out,
                            int32_t max_ctas, int32_t* dev_err, cudaStream_t stream);

/*
 * ple_select_rows -- this replica's token window out of the buffer the
 * group exchanged, heads back in head order, fp8 codes dequantised.
 * (PR#56512 report, 实现拆解 4: _engram_select_rows takes the token window
 * from the rank-major gathered buffer; PR#54371 report, 实现拆解 3:
 * _select_embeddings returns the DP-local rows.)
 *
 *   out[t][h*D + c] = src[p][row_begin + t][k*D + c]                  (bf16)
 *   out[t][h*D + c] = bf16_rn(float(e4m3(src[p][row_begin + t][k*D + c]))
 *                             * src_scale[p][row_begin + t][k])      (fp8)
 * with p = part_of_head[h], k = col_of_head[h], t < num_tokens.
 *
 *   src          [num_parts][part_rows][part_heads * head_dim] device, bf16
 *                (PLE_BF16) or e4m3 codes (either fp8 dtype), 16-byte
 *                aligned: e.g. the all-gathered head-shard outputs of the
 *                group (part = group rank), or the reduced row-shard
 *                outputs (one part).
 *   src_scale    [num_parts][part_rows][part_heads] float32 device (fp8).
 *   part_of_head, col_of_head  host arrays [num_heads]: where head h sits.
 *   out          [num_tokens][num_heads * head_dim] bf16 device, 16-byte
 *                aligned.
 * Errors: a window outside [0, part_rows), a head mapped outside the parts
 * or columns -> PLE_ERR_INVALID_ARG; more than PLE_MAX_HEADS heads, a row
 * that is not a multiple of 16 bytes -> PLE_ERR_UNSUPPORTED.
 */
ple_status ple_select_rows(const void* src, int32_t num_parts, int64_t part_rows,
                           int32_t part_heads, const float* src_scale, int64_t row_begin,
                           int64_t num_tokens, int32_t num_heads, const int32_t* part_of_head,
                           const int32_t* col_of_head, int32_t head_dim, ple_dtype dtype,
                           ple_bf16_t* out, cudaStream_t stream);

/*
 * ple_wait -- make `consumer` wait for `done`.
 *   timeout_ms <= 0: enqueue a device-side wait only (cudaStreamWaitEvent);
 *                    the host does not block.
 *   timeout_ms  > 0: first poll the event from the host for at most
 *                    timeout_ms; if it has not completed, return
 *                    PLE_ERR_TIMEOUT without touching `consumer`; else
 *                    enqueue the device-side wait and return PLE_OK.
 */
ple_status ple_wait(cudaEvent_t done, cudaStream_t consumer, int32_t timeout_ms);

/*
 * ple_ngram_lookup -- ple_ngram_ids and ple_lookup in one kernel: every
 * gathered row's id is hashed where the gather needs it, so the ids make no
 * round trip through memory (the page's two kernels, PR#54517 report
 * 实现拆解 2 and PR#54371 report 实现拆解 1, fused; this split is the
 * library's own). Arguments as in those two calls, with
 *   ids_out   [num_tokens][H] int64 device or NULL: the ids, when wanted.
 *   ngram_context_out, dev_err, max_ctas: as in ple_ngram_ids / ple_lookup.
 * Results are bit for bit those of ple_ngram_ids followed by ple_lookup.
 * Every head's partition [offsets[h], offsets[h] + vocab_sizes[h]) must lie
 * inside the table's rows (checked on the host: PLE_ERR_INVALID_ARG). The
 * rows are read in token order: for a table in host memory beyond ~16 GB use
 * ple_ngram_ids + ple_lookup_ordered instead.
 */
ple_status ple_ngram_lookup(const int32_t* input_ids, int64_t num_tokens,
                            const int32_t* query_start_loc, int32_t num_reqs,
                            const int32_t* ngram_context, int32_t ctx_len,
                            const int64_t* layer_multipliers,
                            const int64_t* vocab_sizes, const int64_t* offsets,
                            int32_t eos_token_id, int32_t heads_per_ngram,
                            const void* table, int64_t table_rows, int32_t head_dim,
                            ple_dtype dtype, const float* row_scale,
                            ple_table_loc loc, ple_bf16_t* out, int64_t* ids_out,
                            int32_t* ngram_context_out, int32_t max_ctas,
                            int32_t* dev_err, cudaStream_t stream);

/*
 * ple_kv_proj -- merged key/value projection, kv = emb @ W^T.
 * (PR#54517 report, 实现拆解 item 1: key_proj and value_proj merged into one
 * MergedColumnParallelLinear.) W = [W_k; W_v]: rows [0, C) give k, rows
 * [C, 2C) give v. fp32 accumulation on the tensor cores, bf16 result
 * (round to nearest even).
 *
 *   emb   [num_tokens][emb_dim] bf16 device, 16-byte aligned.
 *   w     [2 * hidden][emb_dim] bf16 device, 16-byte aligned.
 *   kv    [num_tokens][2 * hidden] bf16 device.
 * emb_dim must be a multiple of 8 and hidden a multiple of 16
 * (else PLE_ERR_UNSUPPORTED).
 */
ple_status ple_kv_proj(const ple_bf16_t* emb, const ple_bf16_t* w,
                       int64_t num_tokens, int32_t emb_dim, int32_t hidden,
                       ple_bf16_t* kv, int32_t* dev_err, cudaStream_t stream);

/*
 * ple_kv_proj_gate -- ple_kv_proj and the reduction half of ple_gate in one
 * kernel: k is never written to memory. Every 256-column key tile of the
 * projection is rounded to bf16 (the values ple_kv_proj would store) and
 * reduced with the same 256 channels of hidden into per-token partial sums
 * of h^2, k^2 and h*k*gamma_h*gamma_k; the tile that completes a token's
 * sums writes the gate scalar (same formula as ple_gate):
 *   gate_out[t] = sigmoid( <rms(h_t) * gamma_h, rms(k_t) * gamma_k> / sqrt(C) ).
 * The value half kv[:, C:2C) is written exactly as ple_kv_proj writes it;
 * the key half kv[:, 0:C) is left untouched. (The pages fuse the PLE kernels,
 * PR#54517 report 实现拆解 items 1 and 2, without giving this split; it is
 * this library's design.)
 *
 *   emb, w, kv       as in ple_kv_proj.
 *   hidden_states    [num_tokens][hidden] bf16, 16-byte aligned.
 *   gamma_h/gamma_k  [hidden] bf16, 16-byte aligned.
 *   gate_out         [num_tokens] float32.
 *   workspace        device scratch of at least
 *                    ple_kv_proj_gate_workspace(num_tokens, hidden) bytes,
 *                    256-byte aligned, ZERO-FILLED by the caller before its
 *                    first use (e.g. one cudaMemset after allocation). Its
 *                    last bytes hold arrival counters (one per 32 tokens, at
 *                    places fixed by workspace_bytes alone); a call that
 *                    completes leaves them zero again, so the workspace is
 *                    reused with no clearing between calls (and no extra
 *                    node in a CUDA graph), for any num_tokens and hidden it
 *                    has room for -- pass the same workspace_bytes every
 *                    time. After a call that raised a PLE_DEVERR_* bit the
 *                    counters may be left non-zero: clear the workspace
 *                    before reusing it. Stale counters never cause an
 *                    out-of-range access, only wrong gate scalars. Calls in
 *                    flight at once must not share a workspace.
 * hidden must be a multiple of 256 (else PLE_ERR_UNSUPPORTED); a smaller
 * workspace -> PLE_ERR_INVALID_ARG. ple_kv_proj_gate_workspace returns 0 for
 * sizes the call rejects.
 */
size_t ple_kv_proj_gate_workspace(int64_t num_tokens, int32_t hidden);
ple_status ple_kv_proj_gate(const ple_bf16_t* emb, const ple_bf16_t* w,
                            int64_t num_tokens, int32_t emb_dim, int32_t hidden,
                            const ple_bf16_t* hidden_states,
                            const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k,
                            float eps, ple_bf16_t* kv, float* gate_out,
                            void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, cudaStream_t stream);

/*
 * ple_gate -- RMSNorm + sigmoid gate ("PLE gating and normalisation",
 * PR#54517 report 实现拆解 item 2; the pages give no formula, this is the
 * reading the library implements):
 *   g_t = sigmoid( <rms(h_t) * gamma_h, rms(k_t) * gamma_k> / sqrt(C) ),
 *   rms(x) = x / sqrt(mean(x^2) + eps),   u_t = bf16_rn(g_t * v_t).
 *
 *   hidden      [num_tokens][C] bf16.   kv [num_tokens][2C] bf16 (k | v).
 *   gamma_h/k   [C] bf16.                out (u) [num_tokens][C] bf16.
 *   gate_out    [num_tokens] float32 or NULL (the scalar gates).
 * C must be a multiple of 8 (else PLE_ERR_INVALID_ARG) and at most 16384
 * (else PLE_ERR_UNSUPPORTED); the same bound holds for ple_gate_conv.
 */
ple_status ple_gate(const ple_bf16_t* hidden, const ple_bf16_t* kv,
                    const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k,
                    float eps, int64_t num_tokens, int32_t hidden_size,
                    ple_bf16_t* out, float* gate_out, cudaStream_t stream);

/*
 * ple_conv -- dilated causal depthwise short conv over ragged requests
 * (PR#54517 report 实现拆解 items 2 and 4: _ple_conv_kernel, prefill and
 * decode with a cached state). For token t of request r, channel c:
 *   y_t[c] = sum_{i<K} w[c][i] * x_{t - (K-1-i)*dilation}[c]
 * over r's virtual sequence conv_state[r] ++ x[segment of r]; positions
 * before it read zeros (conv_state == NULL means all-zero history).
 *
 *   x               [num_tokens][C] bf16.      w [C][K] bf16.
 *   query_start_loc [num_reqs + 1] int32 device (same rules as ple_ngram_ids).
 *   conv_state      [num_reqs][(K-1)*dilation][C] bf16 (history, oldest first)
 *                   or NULL.
 *   conv_state_out  same shape or NULL: the last (K-1)*dilation inputs of
 *                   each virtual sequence. Must not overlap conv_state.
 *   out             [num_tokens][C] bf16.
 * K in 1 .. 8, dilation >= 1, (K-1)*dilation <= 64, C a multiple of 8.
 * The state buffers must be 16-byte aligned.
 */
ple_status ple_conv(const ple_bf16_t* x, const int32_t* query_start_loc,
                    int32_t num_reqs, int64_t num_tokens, int32_t hidden_size,
                    const ple_bf16_t* w, int32_t kernel_size, int32_t dilation,
                    const ple_bf16_t* conv_state, ple_bf16_t* conv_state_out,
                    ple_bf16_t* out, int32_t* dev_err, cudaStream_t stream);

/*
 * ple_gate_conv -- ple_gate followed by ple_conv without materialising u:
 * a reduction pass writes the gate scalars g_t to gate_out (4 bytes per
 * token), then the conv pass stages the dilation window u = bf16_rn(g * v)
 * in shared memory and convolves it; u never reaches global memory. Same
 * results as ple_gate then ple_conv.
 * Arguments as in those two calls; gate_out [num_tokens] float32 is
 * REQUIRED here (it carries g between the two passes), else
 * PLE_ERR_INVALID_ARG.
 */
ple_status ple_gate_conv(const ple_bf16_t* hidden, const ple_bf16_t* kv,
                         const ple_bf16_t* gamma_h, const ple_bf16_t* gamma_k,
                         float eps, const int32_t* query_start_loc,
                         int32_t num_reqs, int64_t num_tokens,
                         int32_t hidden_size, const ple_bf16_t* w,
                         int32_t kernel_size, int32_t dilation,
                         const ple_bf16_t* conv_state,
                         ple_bf16_t* conv_state_out, ple_bf16_t* out,
                         float* gate_out, int32_t* dev_err,
                         cudaStream_t stream);

/*
 * ple_gated_conv -- the conv pass of ple_gate_conv with the gate scalars
 * given (from ple_kv_proj_gate or ple_gate): convolves
 * u_t = bf16_rn(gate[t] * v_t), v_t = kv[t][C:2C), staged in shared memory
 * only. Same results as ple_conv on u.
 *   kv    [num_tokens][2 * hidden_size] bf16 (only the v half is read).
 *   gate  [num_tokens] float32.
 * Other arguments and limits as in ple_conv.
 */
ple_status ple_gated_conv(const ple_bf16_t* kv, const float* gate,
                          const int32_t* query_start_loc, int32_t num_reqs,
                          int64_t num_tokens, int32_t hidden_size,
                          const ple_bf16_t* w, int32_t kernel_size,
                          int32_t dilation, const ple_bf16_t* conv_state,
                          ple_bf16_t* conv_state_out, ple_bf16_t* out,
                          int32_t* dev_err, cudaStream_t stream);

/*
 * ple_host_table_alloc / ple_host_table_free -- host memory for a table read
 * over UVA (PLE_HOST_UVA). (PR#54371 report: the pinned-host backend keeps the
 * weight in pinned memory and the GPU reads the rows it needs in place;
 * PR#56512 report: a mapped table registered with cudaHostRegister.)
 * The memory is an anonymous mapping aligned to 1 GiB, advised for
 * transparent huge pages and registered with cudaHostRegister, so the GPU
 * translates it with huge pages: a random row gather over a multi-GB table
 * then runs near the host-link rate, where cudaHostAlloc memory is bounded by
 * address-translation misses. These are the only entry points that allocate;
 * the caller owns the memory and frees it with the same byte count.
 *   bytes      > 0.    host_ptr   receives the 1 GiB-aligned host address.
 * Errors: mmap failure or cudaHostRegister failure -> PLE_ERR_CUDA
 * (nothing stays allocated).
 */
ple_status ple_host_table_alloc(size_t bytes, void** host_ptr);
ple_status ple_host_table_free(void* host_ptr, size_t bytes);

/* Flags of the shared and file-backed host tables below. */
typedef enum {
  PLE_HOST_TABLE_REGISTER = 1 /* cudaHostRegister the mapping (needed for UVA reads) */
} ple_host_table_flags;

/*
 * ple_host_table_create_shared / ple_host_table_attach_shared /
 * ple_host_table_unlink_shared -- a table in a named POSIX shared-memory
 * object (/dev/shm), mapped MAP_SHARED by several processes and registered
 * with cudaHostRegister so each one's GPU reads it in place over UVA.
 * (PR#56512 report, 关键源码片段: a /dev/shm backing file mapped MAP_SHARED and
 * registered with cudaHostRegister, created by one leader that alone writes
 * the weights, with every step rolled back on failure.)
 *   name        "/" then 1..254 characters without "/", else PLE_ERR_INVALID_ARG.
 *   bytes       > 0; create sizes the object to `bytes` (it must not exist);
 *               attach requires an existing object of at least `bytes`.
 *   flags       PLE_HOST_TABLE_REGISTER to register for GPU reads (0: map only).
 *   host_ptr    receives the mapping (advised for huge pages, NUMA policy set).
 * On any failure everything the call did is undone (mapping, descriptor and,
 * for create, the object itself) and *host_ptr is NULL. The object outlives
 * its mappings until ple_host_table_unlink_shared.
 */
ple_status ple_host_table_create_shared(const char* name, size_t bytes, int32_t flags,
                                        void** host_ptr);
ple_status ple_host_table_attach_shared(const char* name, size_t bytes, int32_t flags,
                                        void** host_ptr);
ple_status ple_host_table_unlink_shared(const char* name);

/*
 * ple_host_table_map_file -- a table stored in a file, mapped read-only
 * (MAP_SHARED, madvise MADV_RANDOM) and, with PLE_HOST_TABLE_REGISTER,
 * registered read-only for GPU reads over UVA (registration pins the pages,
 * reading the file into the page cache). Where read-only registration is
 * not supported the file is mapped privately and registered (each page then
 * gets its own copy in memory; the file is never written). (PR#53899 page:
 * the disk-backed mmap table storage read with MADV_RANDOM.) The file must
 * hold at least `bytes`; on failure nothing stays mapped.
 */
ple_status ple_host_table_map_file(const char* path, size_t bytes, int32_t flags,
                                   void** host_ptr);

/* Undo ple_host_table_create_shared / _attach_shared / _map_file (the same
 * bytes and flags): unregister if registered, then unmap. */
ple_status ple_host_table_unmap(void* host_ptr, size_t bytes, int32_t flags);

/*
 * Step runtime of the end-to-end host path (a layer run over host buffers):
 * graph capture of a step's library calls, and one step enqueued across
 * three caller-created streams so that neighbouring steps overlap --
 *   copy_in   waits `computed`, uploads, records `loaded`;
 *   compute   waits `loaded` and `returned`, runs the step, records `computed`;
 *   copy_out  waits `computed`, reads back, records `returned`.
 * With one set of device buffers and three events per pipeline slot, a
 * slot's inputs are overwritten only after its previous step computed, and
 * its device outputs only after they were read back; an event never
 * recorded counts as complete, so a slot's first step waits for nothing.
 * Host pointers of the copies must be pinned (or registered) for the copies
 * to run asynchronously. Each copy is one cudaMemcpyAsync. (The pages run
 * the layer from Python; this host path is an addition, needed because a
 * small step's host-side launches and waits cost more than its kernels.)
 * The graph and event objects below are the library's only allocations
 * besides ple_host_table_alloc; the caller destroys them.
 */
typedef struct {
  void* dst;        /* device (upload) or host (read-back) */
  const void* src;  /* host (upload) or device (read-back) */
  size_t bytes;     /* 0: skipped */
} ple_copy;

typedef struct ple_graph_s* ple_graph;

/* ple_graph_begin / ple_graph_end -- capture the work the calling thread
 * enqueues on `stream` between the two calls (thread-local capture mode:
 * library calls only; nothing may allocate device memory meanwhile) into an
 * instantiated graph. ple_graph_end always ends the capture; *graph is NULL
 * on failure (a call in between that cannot be captured fails the end). */
ple_status ple_graph_begin(cudaStream_t stream);
ple_status ple_graph_end(cudaStream_t stream, ple_graph* graph);
/* Launch a captured graph on `stream`; destroy one (NULL: no-op). */
ple_status ple_graph_launch(ple_graph graph, cudaStream_t stream);
void ple_graph_destroy(ple_graph graph);

/* Events for the step runtime (timing disabled); ple_event_synchronize
 * blocks the host until `event` completes. Destroy: NULL is a no-op. */
ple_status ple_event_create(cudaEvent_t* event);
void ple_event_destroy(cudaEvent_t event);
ple_status ple_event_synchronize(cudaEvent_t event);

/* ple_step_begin -- the copy-in half of a step (wait `computed`, uploads,
 * record `loaded`) and the compute stream's waits on `loaded` and
 * `returned`; the caller then enqueues the step's work on `compute`.
 * ple_step_end -- record `computed` on `compute`, then the read-backs on
 * `copy_out` after it, then record `returned`. Streams must be distinct and
 * created (not the legacy default stream); null events, a negative copy
 * count or a null pointer of a non-empty copy -> PLE_ERR_INVALID_ARG with
 * nothing enqueued. */
ple_status ple_step_begin(cudaStream_t copy_in, cudaStream_t compute, const ple_copy* uploads,
                          int32_t num_uploads, cudaEvent_t loaded, cudaEvent_t computed,
                          cudaEvent_t returned);
ple_status ple_step_end(cudaStream_t compute, cudaStream_t copy_out, const ple_copy* downloads,
                        int32_t num_downloads, cudaEvent_t computed, cudaEvent_t returned);
/* ple_step -- ple_step_begin, the launch of `graph` on `compute`, then
 * ple_step_end, in one call (same argument rules; `graph` non-NULL). */
ple_status ple_step(cudaStream_t copy_in, cudaStream_t compute, cudaStream_t copy_out,
                    const ple_copy* uploads, int32_t num_uploads, ple_graph graph,
                    const ple_copy* downloads, int32_t num_downloads, cudaEvent_t loaded,
                    cudaEvent_t computed, cudaEvent_t returned);

/* Text of the last non-OK status on this host thread ("" if none). */
const char* ple_last_error(void);

/* Library version string. */
const char* ple_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PLE_H_ */
