// ple_lookup_shard / ple_select_rows: the two kernel steps of a lookup whose
// table is split across the ranks of an exchange group.
//
// Sources: PR#56512 report ("[DS V4.1][Engram] Support async prefetch for
// offloaded engram lookups and engram DP sharding"), 执行摘要 and 实现拆解
// items 3-4: heads sharded over the engram-DP group in TP-major order
// (engram_head_shard_rank), hashes padded and all-gathered across the group
// (gather_engram_hashes), each rank looks up its heads for every gathered
// token, and _engram_select_rows takes this rank's token window from the
// rank-major gathered buffer. PR#54371 report ("[Qwen4Exp] Support UVA
// PLE-offload and Engram tensor parallelism"), 实现拆解 item 3 and
// 关键源码片段 (_get_dp_gather_slot, _gather_dp_ids, _select_embeddings): the
// table sharded over ETP = TP x DP ranks, the DP ids gathered into slots of the
// group's largest token count, the looked-up rows combined across the group
// by a parallel reduce (fp8 rows reduced through an int8 view, test
// test_ple_fp8_embedding_uses_int8_for_parallel_reduce) and this replica's
// slot selected.
//
// ple_lookup_shard gathers the rows one rank owns:
//   head shard (PLE_SHARD_HEADS): the rank's table holds the rows of a range
//     of heads; the output holds those heads' rows (fp8 dequantised), and an
//     id outside the rank's rows is an error (zero row + PLE_DEVERR_BOUNDS).
//   row shard (PLE_SHARD_ROWS): the rank's table holds a contiguous range of
//     the concatenated table's rows; ids outside it give zero bytes (another
//     rank owns them) and the output keeps the table's raw bytes (bf16 bits,
//     or e4m3 codes plus a float32 scale per row), so that summing the ranks'
//     outputs as 8-bit integers -- one nonzero contributor per byte --
//     rebuilds every row exactly.
// ple_select_rows copies (and for fp8 codes dequantises) this replica's token
// window out of the exchanged buffer, putting each head's rows back in head
// order.
//
// Both are HBM-bound copies: one thread per 16-byte vector, kUnroll vectors in
// flight per thread before any store, like the plain gather.
#include "common.cuh"
#include "rows.cuh"

namespace ple {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kMaxSelectHeads = 64;

// OUT_FP8_DEQUANT: fp8 codes in, bf16 out (head shard of an fp8 table).
// Otherwise the row's raw 16-byte vectors are copied (bf16 rows, or fp8
// codes of a row shard, whose scales go to scale_out).
template <bool OUT_FP8_DEQUANT>
__global__ void __launch_bounds__(kThreads)
shard_gather_kernel(const int64_t* __restrict__ ids, int ids_heads, int head_begin, int num_heads,
                    uint32_t total_vecs, int vpr, const uint4* __restrict__ table,
                    const float* __restrict__ row_scale, int scale_stride, int64_t table_rows,
                    int64_t row_base, int rows_mode, uint4* __restrict__ out,
                    float* __restrict__ scale_out, int32_t* dev_err) {
  pdl_wait();
  pdl_trigger();
  const uint32_t step = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total_vecs;
       base += step * kUnroll) {
    uint4 v[kUnroll];
    float s[kUnroll];
    uint32_t o[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * step;
      v[u] = make_uint4(0, 0, 0, 0);
      s[u] = 0.f;
      o[u] = total_vecs;
      if (idx < total_vecs) {
        const uint32_t p = idx / vpr;  // (token, head) item
        const uint32_t k = idx - p * vpr;
        const uint32_t t = p / num_heads;
        const uint32_t j = p - t * num_heads;
        o[u] = idx;
        const int64_t local =
            __ldg(ids + static_cast<int64_t>(t) * ids_heads + head_begin + j) - row_base;
        if (static_cast<uint64_t>(local) < static_cast<uint64_t>(table_rows)) {
          v[u] = load_row_vec(table + local * vpr + k);
          if (row_scale != nullptr) s[u] = __ldg(row_scale + local * scale_stride);
        } else if (!rows_mode) {
          set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // the row is written as zeros
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] >= total_vecs) continue;
      if constexpr (OUT_FP8_DEQUANT) {
        uint4 lo, hi;
        dequant16(v[u], s[u], &lo, &hi);
        out[2 * static_cast<size_t>(o[u])] = lo;
        out[2 * static_cast<size_t>(o[u]) + 1] = hi;
      } else {
        out[o[u]] = v[u];
        if (scale_out != nullptr && o[u] % vpr == 0) scale_out[o[u] / vpr] = s[u];
      }
    }
  }
}

struct SelectMap {
  int32_t part[kMaxSelectHeads];  // exchanged part holding head h
  int32_t col[kMaxSelectHeads];   // head slot of h inside that part
};

// out[t][h] <- src[part(h)][row_begin + t][col(h)] (16-byte vectors; FP8:
// dequantised with the matching entry of src_scale).
template <bool FP8>
__global__ void __launch_bounds__(kThreads)
select_rows_kernel(const uint4* __restrict__ src, int64_t part_vecs, int64_t row_vecs,
                   const float* __restrict__ src_scale, int64_t scale_part, int part_heads,
                   int64_t row_begin, uint32_t total_vecs, int num_heads, int vpr,
                   const __grid_constant__ SelectMap map, uint4* __restrict__ out) {
  // the head map in shared memory: the lanes of a warp index different heads,
  // and a lane-varying index into the parameter block would serialise on the
  // constant cache
  __shared__ int32_t part_s[kMaxSelectHeads], col_s[kMaxSelectHeads];
  for (int h = threadIdx.x; h < num_heads; h += kThreads) {
    part_s[h] = map.part[h];
    col_s[h] = map.col[h];
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const uint32_t step = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total_vecs;
       base += step * kUnroll) {
    uint4 v[kUnroll];
    float s[kUnroll];
    uint32_t o[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * step;
      o[u] = total_vecs;
      s[u] = 0.f;
      v[u] = make_uint4(0, 0, 0, 0);
      if (idx < total_vecs) {
        const uint32_t p = idx / vpr;
        const uint32_t k = idx - p * vpr;
        const uint32_t t = p / num_heads;
        const uint32_t h = p - t * num_heads;
        const int part = part_s[h];
        const int col = col_s[h];
        const int64_t row = row_begin + t;
        o[u] = idx;
        v[u] = __ldg(src + part * part_vecs + row * row_vecs + static_cast<int64_t>(col) * vpr + k);
        if (FP8) s[u] = __ldg(src_scale + part * scale_part + row * part_heads + col);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] >= total_vecs) continue;
      if constexpr (FP8) {
        uint4 lo, hi;
        dequant16(v[u], s[u], &lo, &hi);
        out[2 * static_cast<size_t>(o[u])] = lo;
        out[2 * static_cast<size_t>(o[u]) + 1] = hi;
      } else {
        out[o[u]] = v[u];
      }
    }
  }
}

unsigned copy_grid(int64_t total_vecs, int32_t max_ctas) {
  int64_t blocks = (total_vecs + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int64_t full = static_cast<int64_t>(num_sms()) * (2048 / kThreads);
  if (blocks > full) blocks = full;
  if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_lookup_shard(const int64_t* ids, int64_t num_tokens, int32_t ids_heads,
                                       int32_t head_begin, int32_t num_heads, const void* table,
                                       int64_t table_rows, int64_t row_base, int32_t head_dim,
                                       ple_dtype dtype, const float* row_scale,
                                       ple_table_loc loc, ple_shard_kind kind, void* out,
                                       float* scale_out, int32_t max_ctas, int32_t* dev_err,
                                       cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_lookup_shard";
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1 || table_rows < 0 || row_base < 0 ||
      head_begin < 0 || ids_heads < 1 || head_begin + num_heads > ids_heads)
    return fail(PLE_ERR_INVALID_ARG,
                "%s: bad sizes (T=%lld ids_heads=%d heads [%d, %d) D=%d rows=%lld base=%lld)",
                name, static_cast<long long>(num_tokens), ids_heads, head_begin,
                head_begin + num_heads, head_dim, static_cast<long long>(table_rows),
                static_cast<long long>(row_base));
  if (dtype != PLE_BF16 && dtype != PLE_FP8_E4M3 && dtype != PLE_FP8_E4M3_TENSOR)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown dtype %d", name, static_cast<int>(dtype));
  if (kind != PLE_SHARD_HEADS && kind != PLE_SHARD_ROWS)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown shard kind %d", name, static_cast<int>(kind));
  if (loc != PLE_HBM && loc != PLE_HOST_UVA)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown table location %d", name, static_cast<int>(loc));
  const bool fp8 = dtype != PLE_BF16;
  const int elem = fp8 ? 1 : 2;
  if ((static_cast<int64_t>(head_dim) * elem) % 16 != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: row of %d bytes is not a multiple of 16", name,
                head_dim * elem);
  if (num_tokens == 0) return PLE_OK;
  if (!ids || !table || !out) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (fp8 && !row_scale) return fail(PLE_ERR_INVALID_ARG, "%s: fp8 table needs row_scale", name);
  const bool rows_mode = kind == PLE_SHARD_ROWS;
  if (rows_mode && fp8 && !scale_out)
    return fail(PLE_ERR_INVALID_ARG, "%s: an fp8 row shard needs scale_out", name);
  if (!aligned16(table) || !aligned16(out))
    return fail(PLE_ERR_INVALID_ARG, "%s: table and out must be 16-byte aligned", name);
  cudaPointerAttributes attr{};
  cudaError_t aerr = cudaPointerGetAttributes(&attr, table);
  if (aerr != cudaSuccess) return check_cuda(aerr, "cudaPointerGetAttributes(table)");
  if (loc == PLE_HOST_UVA && attr.type != cudaMemoryTypeHost)
    return fail(PLE_ERR_INVALID_ARG,
                "%s: PLE_HOST_UVA table is not pinned/registered host memory (type %d)", name,
                static_cast<int>(attr.type));
  if (loc == PLE_HBM && attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(PLE_ERR_INVALID_ARG, "%s: PLE_HBM table is not device memory (type %d)", name,
                static_cast<int>(attr.type));
  const int vpr = static_cast<int>(static_cast<int64_t>(head_dim) * elem / 16);
  const int64_t total = num_tokens * num_heads * vpr;
  if (total >= (int64_t(1) << 31))
    return fail(PLE_ERR_UNSUPPORTED, "%s: %lld row vectors exceed one launch", name,
                static_cast<long long>(total));
  const uint4* tab = static_cast<const uint4*>(attr.devicePointer ? attr.devicePointer : table);
  const int scale_stride = dtype == PLE_FP8_E4M3 ? 1 : 0;
  const dim3 grid(copy_grid(total, max_ctas));
  const bool dequant = fp8 && !rows_mode;
  cudaError_t err;
  if (dequant)
    err = launch_kernel(shard_gather_kernel<true>, grid, dim3(kThreads), 0, stream, 1, ids,
                        ids_heads, head_begin, num_heads, static_cast<uint32_t>(total), vpr, tab,
                        row_scale, scale_stride, table_rows, row_base, 0,
                        static_cast<uint4*>(out), static_cast<float*>(nullptr), dev_err);
  else
    err = launch_kernel(shard_gather_kernel<false>, grid, dim3(kThreads), 0, stream, 1, ids,
                        ids_heads, head_begin, num_heads, static_cast<uint32_t>(total), vpr, tab,
                        fp8 ? row_scale : nullptr, scale_stride, table_rows, row_base,
                        rows_mode ? 1 : 0, static_cast<uint4*>(out), fp8 ? scale_out : nullptr,
                        dev_err);
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}

PLE_EXPORT ple_status ple_select_rows(const void* src, int32_t num_parts, int64_t part_rows,
                                      int32_t part_heads, const float* src_scale,
                                      int64_t row_begin, int64_t num_tokens, int32_t num_heads,
                                      const int32_t* part_of_head, const int32_t* col_of_head,
                                      int32_t head_dim, ple_dtype dtype, ple_bf16_t* out,
                                      cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_select_rows";
  if (num_parts < 1 || part_rows < 0 || part_heads < 1 || row_begin < 0 || num_tokens < 0 ||
      num_heads < 1 || head_dim < 1 || row_begin + num_tokens > part_rows)
    return fail(PLE_ERR_INVALID_ARG,
                "%s: bad sizes (parts=%d rows=%lld heads=%d window [%lld, %lld) H=%d D=%d)", name,
                num_parts, static_cast<long long>(part_rows), part_heads,
                static_cast<long long>(row_begin), static_cast<long long>(row_begin + num_tokens),
                num_heads, head_dim);
  if (num_heads > kMaxSelectHeads)
    return fail(PLE_ERR_UNSUPPORTED, "%s: at most %d heads", name, kMaxSelectHeads);
  if (dtype != PLE_BF16 && dtype != PLE_FP8_E4M3 && dtype != PLE_FP8_E4M3_TENSOR)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown dtype %d", name, static_cast<int>(dtype));
  const bool fp8 = dtype != PLE_BF16;
  const int elem = fp8 ? 1 : 2;
  if ((static_cast<int64_t>(head_dim) * elem) % 16 != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: row of %d bytes is not a multiple of 16", name,
                head_dim * elem);
  if (!part_of_head || !col_of_head)
    return fail(PLE_ERR_INVALID_ARG, "%s: null head map", name);
  SelectMap map{};
  for (int h = 0; h < num_heads; ++h) {
    if (part_of_head[h] < 0 || part_of_head[h] >= num_parts || col_of_head[h] < 0 ||
        col_of_head[h] >= part_heads)
      return fail(PLE_ERR_INVALID_ARG, "%s: head %d maps to part %d, column %d", name, h,
                  part_of_head[h], col_of_head[h]);
    map.part[h] = part_of_head[h];
    map.col[h] = col_of_head[h];
  }
  if (num_tokens == 0) return PLE_OK;
  if (!src || !out || (fp8 && !src_scale))
    return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(src) || !aligned16(out))
    return fail(PLE_ERR_INVALID_ARG, "%s: src and out must be 16-byte aligned", name);
  const int vpr = static_cast<int>(static_cast<int64_t>(head_dim) * elem / 16);
  const int64_t total = num_tokens * num_heads * vpr;
  if (total >= (int64_t(1) << 31))
    return fail(PLE_ERR_UNSUPPORTED, "%s: %lld vectors exceed one launch", name,
                static_cast<long long>(total));
  const int64_t row_vecs = static_cast<int64_t>(part_heads) * vpr;
  const int64_t part_vecs = part_rows * row_vecs;
  const dim3 grid(copy_grid(total, 0));
  cudaError_t err;
  if (fp8)
    err = launch_kernel(select_rows_kernel<true>, grid, dim3(kThreads), 0, stream, 1,
                        static_cast<const uint4*>(src), part_vecs, row_vecs, src_scale,
                        part_rows * part_heads, part_heads, row_begin,
                        static_cast<uint32_t>(total), num_heads, vpr, map,
                        reinterpret_cast<uint4*>(out));
  else
    err = launch_kernel(select_rows_kernel<false>, grid, dim3(kThreads), 0, stream, 1,
                        static_cast<const uint4*>(src), part_vecs, row_vecs,
                        static_cast<const float*>(nullptr), int64_t(0), part_heads, row_begin,
                        static_cast<uint32_t>(total), num_heads, vpr, map,
                        reinterpret_cast<uint4*>(out));
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}
