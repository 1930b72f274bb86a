// ple_lookup / ple_lookup_prefetch: multi-head row gather from a PLE table in
// HBM or in pinned host memory (UVA), bf16 rows or fp8 e4m3 rows with a
// per-row float32 scale dequantised on the fly.
//
// Sources: PR#54371 report ("Support UVA PLE-offload ..."), 实现拆解 item 1 and
// 关键源码片段 (Qwen4ExpPLEDeviceEmbedding / Qwen4ExpPLEPinnedHostEmbedding:
// F.embedding over a device table or over a pinned host table read in place
// through UVA; start_prefetch on a prefetch stream; BF16 / FP8 weight
// methods). PR#56512 report, 实现拆解 item 4 (side-stream lookup with a
// reduced grid). PR#53899 page (FP8 table with a weight_scale).
//
// Design (HBM-bound, no tensor cores): the output is a flat array of 16-byte
// vectors. A work item is one output vector; consecutive threads take
// consecutive vectors, so the threads of a row read one contiguous table row
// (256 B for D = 128 bf16: 16 threads) and write one contiguous output slice.
// Each thread issues UNROLL independent row loads before any store to keep
// enough bytes in flight (HBM: ~64 KB per SM; host link: more, hence the
// unroll). Table reads bypass L1 (ld.global.nc.L1::no_allocate) and ask L2 for
// the whole 256-B row; output stores are ordinary write-back stores so that
// the next kernel (kv_proj) finds the rows in L2.
#include "common.cuh"

#include <cuda_fp8.h>

namespace ple {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 load_row_vec(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// bf16 rows: VPR = 16-byte vectors per row (template for the common sizes,
// 0 = runtime value).
template <int VPR>
__global__ void __launch_bounds__(kThreads)
gather_bf16_kernel(const int64_t* __restrict__ ids, uint32_t total_vecs, int vpr_rt,
                   const uint4* __restrict__ table, int64_t table_rows,
                   uint4* __restrict__ out, int32_t* dev_err) {
  const int vpr = VPR ? VPR : vpr_rt;
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total_vecs;
       base += stride * kUnroll) {
    uint4 v[kUnroll];
    uint32_t idx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      idx[u] = base + u * stride;
      v[u] = make_uint4(0, 0, 0, 0);
      if (idx[u] < total_vecs) {
        const uint32_t row_out = idx[u] / vpr;  // (token, head) pair
        const uint32_t k = idx[u] - row_out * vpr;
        const int64_t id = __ldg(ids + row_out);
        if (static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows)) {
          v[u] = load_row_vec(table + id * vpr + k);
        } else {
          set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // the row is written as zeros
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (idx[u] < total_vecs) out[idx[u]] = v[u];
  }
}

// fp8 rows: each work item is 16 codes (one 16-byte load) -> 16 bf16 values
// (two 16-byte stores). VPR = code vectors per row.
__device__ __forceinline__ uint32_t dequant_pair(uint16_t codes, float scale) {
  const __half2 h2(__nv_cvt_fp8x2_to_halfraw2(codes, __NV_E4M3));
  const float2 f = __half22float2(h2);
  const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
  return *reinterpret_cast<const uint32_t*>(&b);
}

__device__ __forceinline__ void dequant16(uint4 c, float s, uint4* lo, uint4* hi) {
  lo->x = dequant_pair(static_cast<uint16_t>(c.x & 0xFFFF), s);
  lo->y = dequant_pair(static_cast<uint16_t>(c.x >> 16), s);
  lo->z = dequant_pair(static_cast<uint16_t>(c.y & 0xFFFF), s);
  lo->w = dequant_pair(static_cast<uint16_t>(c.y >> 16), s);
  hi->x = dequant_pair(static_cast<uint16_t>(c.z & 0xFFFF), s);
  hi->y = dequant_pair(static_cast<uint16_t>(c.z >> 16), s);
  hi->z = dequant_pair(static_cast<uint16_t>(c.w & 0xFFFF), s);
  hi->w = dequant_pair(static_cast<uint16_t>(c.w >> 16), s);
}

template <int VPR>
__global__ void __launch_bounds__(kThreads)
gather_fp8_kernel(const int64_t* __restrict__ ids, uint32_t total_vecs, int vpr_rt,
                  const uint4* __restrict__ table, const float* __restrict__ row_scale,
                  int64_t table_rows, uint4* __restrict__ out, int32_t* dev_err) {
  const int vpr = VPR ? VPR : vpr_rt;
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total_vecs;
       base += stride * kUnroll) {
    uint4 c[kUnroll];
    float s[kUnroll];
    uint32_t idx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      idx[u] = base + u * stride;
      c[u] = make_uint4(0, 0, 0, 0);
      s[u] = 0.f;
      if (idx[u] < total_vecs) {
        const uint32_t row_out = idx[u] / vpr;
        const uint32_t k = idx[u] - row_out * vpr;
        const int64_t id = __ldg(ids + row_out);
        if (static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows)) {
          c[u] = load_row_vec(table + id * vpr + k);
          s[u] = __ldg(row_scale + id);
        } else {
          set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // the row is written as zeros
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (idx[u] < total_vecs) {
        uint4 lo, hi;
        dequant16(c[u], s[u], &lo, &hi);
        out[2 * static_cast<size_t>(idx[u])] = lo;
        out[2 * static_cast<size_t>(idx[u]) + 1] = hi;
      }
    }
  }
}

ple_status launch_gather(const int64_t* ids, int64_t num_tokens, int32_t num_heads,
                         const void* table, int64_t table_rows, int32_t head_dim,
                         ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                         ple_bf16_t* out, int32_t max_ctas, int32_t* dev_err,
                         cudaStream_t stream, const char* name) {
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1 || table_rows < 0)
    return fail(PLE_ERR_INVALID_ARG, "%s: bad sizes (T=%lld H=%d D=%d rows=%lld)", name,
                static_cast<long long>(num_tokens), num_heads, head_dim,
                static_cast<long long>(table_rows));
  if (dtype != PLE_BF16 && dtype != PLE_FP8_E4M3)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown dtype %d", name, static_cast<int>(dtype));
  if (loc != PLE_HBM && loc != PLE_HOST_UVA)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown table location %d", name, static_cast<int>(loc));
  const int elem = (dtype == PLE_BF16) ? 2 : 1;
  if ((static_cast<int64_t>(head_dim) * elem) % 16 != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: row of %d bytes is not a multiple of 16", name,
                head_dim * elem);
  if (num_tokens == 0) return PLE_OK;
  if (!ids || !table || !out) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (dtype == PLE_FP8_E4M3 && !row_scale)
    return fail(PLE_ERR_INVALID_ARG, "%s: fp8 table needs row_scale", name);
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
  const uint32_t total_vecs = static_cast<uint32_t>(total);
  int64_t blocks = (total + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int64_t full_grid = static_cast<int64_t>(num_sms()) * (2048 / kThreads);
  if (blocks > full_grid) blocks = full_grid;
  if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
  const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : blocks);
  // Read the table through the device view of the allocation (identical to
  // the host address under unified addressing, but ask rather than assume).
  const void* dev_table = attr.devicePointer ? attr.devicePointer : table;
  const uint4* tab = static_cast<const uint4*>(dev_table);
  uint4* o = reinterpret_cast<uint4*>(out);
  if (dtype == PLE_BF16) {
    if (vpr == 16)
      gather_bf16_kernel<16><<<grid, kThreads, 0, stream>>>(ids, total_vecs, vpr, tab, table_rows, o, dev_err);
    else if (vpr == 8)
      gather_bf16_kernel<8><<<grid, kThreads, 0, stream>>>(ids, total_vecs, vpr, tab, table_rows, o, dev_err);
    else
      gather_bf16_kernel<0><<<grid, kThreads, 0, stream>>>(ids, total_vecs, vpr, tab, table_rows, o, dev_err);
  } else {
    if (vpr == 8)
      gather_fp8_kernel<8><<<grid, kThreads, 0, stream>>>(ids, total_vecs, vpr, tab, row_scale, table_rows, o, dev_err);
    else
      gather_fp8_kernel<0><<<grid, kThreads, 0, stream>>>(ids, total_vecs, vpr, tab, row_scale, table_rows, o, dev_err);
  }
  return check_cuda(cudaGetLastError(), name);
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_lookup(const int64_t* ids, int64_t num_tokens, int32_t num_heads,
                                 const void* table, int64_t table_rows, int32_t head_dim,
                                 ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                                 ple_bf16_t* out, int32_t max_ctas, int32_t* dev_err,
                                 cudaStream_t stream) {
  return ple::launch_gather(ids, num_tokens, num_heads, table, table_rows, head_dim, dtype,
                            row_scale, loc, out, max_ctas, dev_err, stream, "ple_lookup");
}

PLE_EXPORT ple_status ple_lookup_prefetch(const int64_t* ids, int64_t num_tokens,
                                          int32_t num_heads, const void* table,
                                          int64_t table_rows, int32_t head_dim,
                                          ple_dtype dtype, const float* row_scale,
                                          ple_table_loc loc, ple_bf16_t* out,
                                          int32_t max_ctas, int32_t* dev_err,
                                          cudaStream_t side_stream, cudaEvent_t done) {
  if (done == nullptr)
    return ple::fail(PLE_ERR_INVALID_ARG, "ple_lookup_prefetch: null event");
  ple_status s = ple::launch_gather(ids, num_tokens, num_heads, table, table_rows, head_dim,
                                    dtype, row_scale, loc, out, max_ctas, dev_err, side_stream,
                                    "ple_lookup_prefetch");
  if (s != PLE_OK) return s;
  return ple::check_cuda(cudaEventRecord(done, side_stream), "ple_lookup_prefetch: record");
}
