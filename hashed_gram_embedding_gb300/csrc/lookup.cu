// ple_lookup / ple_lookup_prefetch / ple_lookup_ordered / ple_ngram_lookup:
// multi-head row gather from a PLE table in HBM or in pinned host memory
// (UVA), bf16 rows or fp8 e4m3 rows with a per-row or whole-table float32
// scale dequantised on the fly; ple_ngram_lookup also hashes the ids.
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
// the next kernel (kv_proj) finds the rows in L2. ple_lookup_ordered walks
// the items in table order (see the page-ordered walk below).
#include "common.cuh"
#include "ngram_hash.cuh"
#include "rows.cuh"

#include <atomic>
#include <cstdlib>
#include <cstring>

namespace ple {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// bf16 rows: VPR = 16-byte vectors per row (template for the common sizes,
// 0 = runtime value).
template <int VPR>
__global__ void __launch_bounds__(kThreads)
gather_bf16_kernel(const int64_t* __restrict__ ids, const uint32_t* __restrict__ perm,
                   uint32_t total_vecs, int vpr_rt, const uint4* __restrict__ table,
                   int64_t table_rows, uint4* __restrict__ out, int32_t* dev_err) {
  pdl_wait();
  // The sorted walk over a host table does not let the next kernel launch
  // early: kernels resident alongside it slow the walk's host reads (measured
  // 3x on a GB300).
  if (perm == nullptr) pdl_trigger();
  const int vpr = VPR ? VPR : vpr_rt;
  // Unsorted walk: a thread's items are a grid apart (all CTAs sweep the
  // whole output together). Sorted walk (perm): a CTA takes kUnroll * 256
  // consecutive items at a time, so the rows in flight at any moment are a
  // narrow slice of the table.
  const uint32_t item_step = perm != nullptr ? kThreads : gridDim.x * kThreads;
  const uint32_t first = perm != nullptr ? blockIdx.x * kThreads * kUnroll + threadIdx.x
                                         : blockIdx.x * kThreads + threadIdx.x;
  const uint32_t iter_step = gridDim.x * kThreads * kUnroll;
  for (uint32_t base = first; base < total_vecs; base += iter_step) {
    uint4 v[kUnroll];
    uint32_t o[kUnroll];  // output vector of each work item
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * item_step;
      v[u] = make_uint4(0, 0, 0, 0);
      o[u] = total_vecs;
      if (idx < total_vecs) {
        const uint32_t p = idx / vpr;  // position in the walk
        const uint32_t k = idx - p * vpr;
        const uint32_t row_out = perm != nullptr ? __ldg(perm + p) : p;  // (token, head) pair
        if (row_out >= total_vecs / vpr) continue;  // (never, for a walk order from the sort)
        o[u] = row_out * vpr + k;
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
      if (o[u] < total_vecs) out[o[u]] = v[u];
  }
}

// fp8 rows: each work item is 16 codes (one 16-byte load) -> 16 bf16 values
// (two 16-byte stores, dequant16). VPR = code vectors per row.
template <int VPR>
__global__ void __launch_bounds__(kThreads)
gather_fp8_kernel(const int64_t* __restrict__ ids, const uint32_t* __restrict__ perm,
                  uint32_t total_vecs, int vpr_rt, const uint4* __restrict__ table,
                  const float* __restrict__ row_scale, int scale_stride, int64_t table_rows,
                  uint4* __restrict__ out, int32_t* dev_err) {
  pdl_wait();
  // The sorted walk over a host table does not let the next kernel launch
  // early: kernels resident alongside it slow the walk's host reads (measured
  // 3x on a GB300).
  if (perm == nullptr) pdl_trigger();
  const int vpr = VPR ? VPR : vpr_rt;
  const uint32_t item_step = perm != nullptr ? kThreads : gridDim.x * kThreads;
  const uint32_t first = perm != nullptr ? blockIdx.x * kThreads * kUnroll + threadIdx.x
                                         : blockIdx.x * kThreads + threadIdx.x;
  const uint32_t iter_step = gridDim.x * kThreads * kUnroll;
  for (uint32_t base = first; base < total_vecs; base += iter_step) {
    uint4 c[kUnroll];
    float s[kUnroll];
    uint32_t o[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * item_step;
      c[u] = make_uint4(0, 0, 0, 0);
      s[u] = 0.f;
      o[u] = total_vecs;
      if (idx < total_vecs) {
        const uint32_t p = idx / vpr;
        const uint32_t k = idx - p * vpr;
        const uint32_t row_out = perm != nullptr ? __ldg(perm + p) : p;
        if (row_out >= total_vecs / vpr) continue;  // (never, for a walk order from the sort)
        o[u] = row_out * vpr + k;
        const int64_t id = __ldg(ids + row_out);
        if (static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows)) {
          c[u] = load_row_vec(table + id * vpr + k);
          s[u] = __ldg(row_scale + id * scale_stride);  // stride 0: one scale for the table
        } else {
          set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // the row is written as zeros
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] < total_vecs) {
        uint4 lo, hi;
        dequant16(c[u], s[u], &lo, &hi);
        out[2 * static_cast<size_t>(o[u])] = lo;
        out[2 * static_cast<size_t>(o[u]) + 1] = hi;
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Token-major gather (the default for a table in HBM): a warp takes tpw
// tokens at a time (tpw * H <= 32). Lane l loads id l of the group (one
// coalesced load for all of the group's heads), then every lane issues all of
// its row-vector loads -- vector j = lane + 32 i of the group's tpw*H*VPR
// vectors, so the 16 (8) lanes of a half (quarter) warp read one whole
// 256-byte (128-byte) row -- before any store. The group's rows are thus in
// flight after one id round trip instead of one round trip per vector (the
// vector-strided kernel above), and the next group's ids are loaded while
// they fly. fp8 rows: lane l reads the scale of item l, shared by shuffle.
// ---------------------------------------------------------------------------
constexpr int kTokLoads = 8;  // row vectors in flight per lane

template <int VPR, bool FP8>
__global__ void __launch_bounds__(kThreads, FP8 ? 3 : 4)
gather_tok_kernel(const int64_t* __restrict__ ids, int64_t T, int H, int tpw,
                  const uint4* __restrict__ table, const float* __restrict__ row_scale,
                  int scale_stride, int64_t table_rows, uint4* __restrict__ out,
                  int32_t* dev_err) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (kThreads / 32) * tpw;
  auto group_id = [&](int64_t t0) {  // id of item `lane` of the group at t0 (-1: none)
    const int64_t n = (T - t0 < tpw ? T - t0 : tpw) * H;
    return lane < n ? __ldg(ids + t0 * H + lane) : int64_t(-1);
  };
  int64_t t0 = warp * tpw;
  int64_t idn = t0 < T ? group_id(t0) : -1;
  for (; t0 < T; t0 += step) {
    const int64_t my_id = idn;
    const int nv = static_cast<int>((T - t0 < tpw ? T - t0 : tpw) * H * VPR);
    if (lane < nv / VPR && static_cast<uint64_t>(my_id) >= static_cast<uint64_t>(table_rows))
      set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // that row is written as zeros
    uint4 v[kTokLoads];
#pragma unroll
    for (int i = 0; i < kTokLoads; ++i) {
      const int j = lane + 32 * i;
      const int item = j / VPR;
      const int64_t id = __shfl_sync(0xffffffffu, my_id, item & 31);
      v[i] = make_uint4(0, 0, 0, 0);
      if (j < nv && static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows))
        v[i] = load_row_vec(table + id * VPR + (j - item * VPR));
    }
    // fp8: lane l reads the scale of item l once; the vectors take it by shuffle
    float my_sc = 0.f;
    if (FP8 && static_cast<uint64_t>(my_id) < static_cast<uint64_t>(table_rows))
      my_sc = __ldg(row_scale + my_id * scale_stride);
    if (t0 + step < T) idn = group_id(t0 + step);  // next group's ids, while the rows fly
    const int64_t o0 = t0 * H * VPR;
#pragma unroll
    for (int i = 0; i < kTokLoads; ++i) {
      const int j = lane + 32 * i;
      if constexpr (FP8) {
        const float sc = __shfl_sync(0xffffffffu, my_sc, (j / VPR) & 31);
        if (j >= nv) continue;
        uint4 lo, hi;
        dequant16(v[i], sc, &lo, &hi);
        out[2 * (o0 + j)] = lo;
        out[2 * (o0 + j) + 1] = hi;
      } else {
        if (j >= nv) continue;
        out[o0 + j] = v[i];
      }
    }
  }
}

// Tokens per warp group for the token-major gather, or 0 when the shape does
// not fit it (more than 32 heads, or more than 32 * kTokLoads row vectors per
// token).
int tok_group(int H, int vpr) {
  if (H < 1 || H > 32 || H * vpr > 32 * kTokLoads) return 0;
  int tpw = 32 / H;
  const int by_loads = 32 * kTokLoads / (H * vpr);
  return tpw < by_loads ? tpw : by_loads;
}

// ---------------------------------------------------------------------------
// ple_ngram_lookup: the n-gram ids and the row gather in one kernel. Each work
// item (one 16-byte table vector of one (token, head) row) hashes its row's
// id itself (ngram_id, request boundaries staged in shared memory, the few
// token loads hitting L1) where the plain gather would load it, so the ids
// never make a round trip through memory; the first vector of each row also
// stores the id when ids_out is given. The walk is the unsorted gather's.
// ---------------------------------------------------------------------------
struct NgramArgs {
  const int32_t* input_ids;
  int64_t num_tokens;
  const int32_t* qsl;
  int num_reqs;
  const int32_t* ctx;
  int ctx_len;
  int eos;
  int heads_per_ngram;
  int num_heads;
  int32_t* ctx_out;
  int64_t* ids_out;
};

template <int VPR, bool FP8>
__global__ void __launch_bounds__(kThreads, 2048 / kThreads)  // the plain gather's full grid
ngram_gather_kernel(const __grid_constant__ NgramArgs na, const __grid_constant__ NgramConsts k,
                    uint32_t total_vecs, int vpr_rt, const uint4* __restrict__ table,
                    const float* __restrict__ row_scale, int scale_stride, int64_t table_rows,
                    uint4* __restrict__ out, int32_t* dev_err) {
  __shared__ int32_t qsl_s[kStagedBounds];
  __shared__ NgramHeadsSmem hs;
  const int R = na.num_reqs;
  const bool staged = R < kStagedBounds;
  stage_ngram_heads(k, na.num_heads, hs);
  pdl_wait();
  pdl_trigger();
  if (staged)
    for (int r = threadIdx.x; r <= R; r += kThreads) qsl_s[r] = __ldg(na.qsl + r);
  __syncthreads();
  const uint32_t gid = blockIdx.x * kThreads + threadIdx.x;
  const uint32_t gsize = gridDim.x * kThreads;
  for (uint32_t i = gid; i <= static_cast<uint32_t>(R); i += gsize)
    check_qsl(na.qsl, R, na.num_tokens, i, dev_err);
  if (na.ctx_out != nullptr)
    for (uint32_t i = gid; i < static_cast<uint32_t>(R) * static_cast<uint32_t>(na.ctx_len);
         i += gsize)
      ngram_carry(na.input_ids, na.num_tokens, na.qsl, R, na.ctx, na.ctx_len, na.eos, i,
                  na.ctx_out);

  const int vpr = VPR ? VPR : vpr_rt;
  const uint32_t H = static_cast<uint32_t>(na.num_heads);
  const int lane = threadIdx.x & 31;
  // The vpr lanes that read one row share its id: with at least kUnroll of
  // them (and rows aligned to the warp), lane j of a row's group hashes the
  // group's row of unrolled step j and passes it on by shuffle; else every
  // lane hashes its own rows.
  const bool shared_ids = vpr >= kUnroll && 32 % vpr == 0;
  auto hash_row = [&](uint32_t p) -> int64_t {  // id of (token, head) row p
    const uint32_t t32 = p / H;
    const int h = static_cast<int>(p - t32 * H);
    const int64_t t = t32;
    // last request whose start is <= t, clamped (as ple_ngram_ids)
    int r;
    int64_t start;
    if (staged) {
      int lo = 0, hi = R + 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(qsl_s[mid]) <= t) lo = mid + 1; else hi = mid;
      }
      r = lo - 1 < 0 ? 0 : (lo - 1 >= R ? R - 1 : lo - 1);
      start = qsl_s[r];
    } else {
      r = find_request(na.qsl, R, t);
      start = __ldg(na.qsl + r);
    }
    return ngram_id(na.input_ids, na.ctx, na.ctx_len, na.eos, t, t - start, r, h,
                    na.heads_per_ngram, k, hs);
  };
  // warp-uniform loop (the shuffles need every lane)
  for (uint32_t wbase = gid - lane; wbase < total_vecs; wbase += gsize * kUnroll) {
    const uint32_t base = wbase + lane;
    int64_t id[kUnroll];
    if (shared_ids) {
      const int g = lane % vpr;  // my place in my row group
      int64_t mine = -1;
      if (g < kUnroll) {
        const uint32_t idx = base - g + g * gsize;  // first vector of step g's row
        if (idx < total_vecs) mine = hash_row(idx / vpr);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) id[u] = __shfl_sync(0xffffffffu, mine, lane - g + u);
    } else {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t idx = base + u * gsize;
        id[u] = idx < total_vecs ? hash_row(idx / vpr) : -1;
      }
    }
    if (na.ids_out != nullptr) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t idx = base + u * gsize;
        if (idx < total_vecs && idx % vpr == 0) na.ids_out[idx / vpr] = id[u];
      }
    }
    uint4 c[kUnroll];
    float sc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {  // their table vectors, all in flight
      const uint32_t idx = base + u * gsize;
      c[u] = make_uint4(0, 0, 0, 0);
      sc[u] = 0.f;
      if (idx < total_vecs) {
        const uint32_t p = idx / vpr;
        if (static_cast<uint64_t>(id[u]) < static_cast<uint64_t>(table_rows)) {
          c[u] = load_row_vec(table + id[u] * vpr + (idx - p * vpr));
          if constexpr (FP8) sc[u] = __ldg(row_scale + id[u] * scale_stride);
        } else {
          set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // the row is written as zeros
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * gsize;
      if (idx >= total_vecs) continue;
      if constexpr (FP8) {
        uint4 lo, hi;
        dequant16(c[u], sc[u], &lo, &hi);
        out[2 * static_cast<size_t>(idx)] = lo;
        out[2 * static_cast<size_t>(idx) + 1] = hi;
      } else {
        out[idx] = c[u];
      }
    }
  }
}


// Token-major ple_ngram_lookup (the default where the shape fits it, as
// gather_tok_kernel): lane l of a warp group hashes the id of item l of the
// group's tpw tokens (ngram_id, request found in the staged boundaries) and
// the group's rows are then loaded as in gather_tok_kernel; the next group's
// ids are hashed while the rows fly.
template <int VPR, bool FP8>
__global__ void __launch_bounds__(kThreads, FP8 ? 3 : 4)
ngram_tok_kernel(const __grid_constant__ NgramArgs na, const __grid_constant__ NgramConsts k,
                 int tpw, const uint4* __restrict__ table, const float* __restrict__ row_scale,
                 int scale_stride, int64_t table_rows, uint4* __restrict__ out,
                 int32_t* dev_err) {
  __shared__ int32_t qsl_s[kStagedBounds];
  __shared__ NgramHeadsSmem hs;
  const int R = na.num_reqs;
  const int H = na.num_heads;
  const int64_t T = na.num_tokens;
  const bool staged = R < kStagedBounds;
  stage_ngram_heads(k, H, hs);
  pdl_wait();
  pdl_trigger();
  if (staged)
    for (int r = threadIdx.x; r <= R; r += kThreads) qsl_s[r] = __ldg(na.qsl + r);
  __syncthreads();
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t gsize = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = gid; i <= R; i += gsize) check_qsl(na.qsl, R, T, i, dev_err);
  if (na.ctx_out != nullptr)
    for (int64_t i = gid; i < static_cast<int64_t>(R) * na.ctx_len; i += gsize)
      ngram_carry(na.input_ids, T, na.qsl, R, na.ctx, na.ctx_len, na.eos, i, na.ctx_out);

  const int lane = threadIdx.x & 31;
  const int64_t warp = gid >> 5;
  const int64_t step = (gsize >> 5) * tpw;
  auto group_id = [&](int64_t t0) -> int64_t {  // hashed id of item `lane` of the group
    const int64_t n = (T - t0 < tpw ? T - t0 : tpw) * H;
    if (lane >= n) return -1;
    const int64_t t = t0 + lane / H;
    const int h = lane - (lane / H) * H;
    int r;
    int64_t start;
    if (staged) {
      int lo = 0, hi = R + 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(qsl_s[mid]) <= t) lo = mid + 1; else hi = mid;
      }
      r = lo - 1 < 0 ? 0 : (lo - 1 >= R ? R - 1 : lo - 1);
      start = qsl_s[r];
    } else {
      r = find_request(na.qsl, R, t);
      start = __ldg(na.qsl + r);
    }
    const int64_t id = ngram_id(na.input_ids, na.ctx, na.ctx_len, na.eos, t, t - start, r, h,
                                na.heads_per_ngram, k, hs);
    if (na.ids_out != nullptr) na.ids_out[t0 * H + lane] = id;
    return id;
  };
  int64_t t0 = warp * tpw;
  int64_t idn = t0 < T ? group_id(t0) : -1;
  for (; t0 < T; t0 += step) {
    const int64_t my_id = idn;
    const int nv = static_cast<int>((T - t0 < tpw ? T - t0 : tpw) * H * VPR);
    if (lane < nv / VPR && static_cast<uint64_t>(my_id) >= static_cast<uint64_t>(table_rows))
      set_dev_err(dev_err, PLE_DEVERR_BOUNDS);  // that row is written as zeros
    uint4 v[kTokLoads];
#pragma unroll
    for (int i = 0; i < kTokLoads; ++i) {
      const int j = lane + 32 * i;
      const int item = j / VPR;
      const int64_t id = __shfl_sync(0xffffffffu, my_id, item & 31);
      v[i] = make_uint4(0, 0, 0, 0);
      if (j < nv && static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows))
        v[i] = load_row_vec(table + id * VPR + (j - item * VPR));
    }
    // fp8: lane l reads the scale of item l once; the vectors take it by shuffle
    float my_sc = 0.f;
    if (FP8 && static_cast<uint64_t>(my_id) < static_cast<uint64_t>(table_rows))
      my_sc = __ldg(row_scale + my_id * scale_stride);
    if (t0 + step < T) idn = group_id(t0 + step);  // next group's ids, while the rows fly
    const int64_t o0 = t0 * H * VPR;
#pragma unroll
    for (int i = 0; i < kTokLoads; ++i) {
      const int j = lane + 32 * i;
      if constexpr (FP8) {
        const float sc = __shfl_sync(0xffffffffu, my_sc, (j / VPR) & 31);
        if (j >= nv) continue;
        uint4 lo, hi;
        dequant16(v[i], sc, &lo, &hi);
        out[2 * (o0 + j)] = lo;
        out[2 * (o0 + j) + 1] = hi;
      } else {
        if (j >= nv) continue;
        out[o0 + j] = v[i];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Bulk-copy gather (bf16 rows, table in HBM). The copy engine moves the rows:
// a warp takes a token, each lane one of its heads, and every lane issues one
// 1-D bulk copy of its row (table -> shared memory) completing on the token's
// mbarrier; once all rows are in, lane 0 writes the token's H*D output values
// (contiguous) back with one bulk store. Each warp keeps kBgSlots tokens in
// flight, so a CTA holds 64 KB of row requests with a few registers per thread
// (the register-fed kernel above is bounded by the registers its in-flight
// loads occupy). Ids outside the table give zero rows written by the lane.
// ---------------------------------------------------------------------------
constexpr int kBgWarps = 4;
constexpr int kBgSlots = 4;
constexpr size_t kBgSmemBudget = 200 * 1024;

__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(kBgWarps * 32)
gather_bulk_kernel(const int64_t* __restrict__ ids, int64_t T, int H, int row_bytes,
                   const uint8_t* __restrict__ table, int64_t table_rows, uint8_t* __restrict__ out,
                   int32_t* dev_err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint32_t tok_bytes = static_cast<uint32_t>(H) * row_bytes;
  uint8_t* slots = smem + static_cast<size_t>(warp) * kBgSlots * tok_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kBgWarps) * kBgSlots * tok_bytes) +
                   warp * kBgSlots;
  if (lane == 0) {
    for (int i = 0; i < kBgSlots; ++i) mbar_init(smem_u32(bars + i), 1);
    mbar_fence_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_trigger();

  const int64_t ta = T * blockIdx.x / gridDim.x;
  const int64_t tb = T * (blockIdx.x + 1) / gridDim.x;
  const int64_t n_my = tb - ta > warp ? (tb - ta - warp + kBgWarps - 1) / kBgWarps : 0;
  auto token = [&](int64_t k) { return ta + warp + k * kBgWarps; };

  // all lanes: start the row copies of token k into its slot
  auto issue = [&](int64_t k) {
    const int64_t t = token(k);
    const int sl = static_cast<int>(k % kBgSlots);
    const uint32_t bar = smem_u32(bars + sl);
    uint8_t* slot = slots + static_cast<size_t>(sl) * tok_bytes;
    int valid = 0;
    for (int h0 = 0; h0 < H; h0 += 32) {
      const int h = h0 + lane;
      bool ok = false;
      int64_t id = 0;
      if (h < H) {
        id = __ldg(ids + t * H + h);
        ok = static_cast<uint64_t>(id) < static_cast<uint64_t>(table_rows);
      }
      valid += __popc(__ballot_sync(0xffffffffu, ok));
      if (h < H && !ok) {  // zero row + flag; ordered before the bulk store below
        uint4* z = reinterpret_cast<uint4*>(slot + static_cast<size_t>(h) * row_bytes);
        for (int q = 0; q < row_bytes / 16; ++q) z[q] = make_uint4(0, 0, 0, 0);
        set_dev_err(dev_err, PLE_DEVERR_BOUNDS);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      if (ok)
        bulk_copy_g2s(smem_u32(slot + static_cast<size_t>(h) * row_bytes),
                      table + id * row_bytes, static_cast<uint32_t>(row_bytes), bar);
    }
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(valid) * row_bytes);
  };

  for (int64_t k = 0; k < n_my && k < kBgSlots; ++k) issue(k);
  int64_t k = 0;
  for (; k < n_my; ++k) {
    const int sl = static_cast<int>(k % kBgSlots);
    const uint32_t parity = static_cast<uint32_t>((k / kBgSlots) & 1);
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(bars + sl), parity, nullptr))) {
      if (lane == 0) set_dev_err(dev_err, PLE_DEVERR_TIMEOUT);
      break;
    }
    __syncwarp();
    if (lane == 0) {
      bulk_store_s2g(out + token(k) * tok_bytes,
                     smem_u32(slots + static_cast<size_t>(sl) * tok_bytes), tok_bytes);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // all but the store just issued have read their slot
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    }
    __syncwarp();
    // refill the slot of token k-1 (its store has read it) with token k-1+S
    if (k >= 1 && k - 1 + kBgSlots < n_my) issue(k - 1 + kBgSlots);
  }
  if (lane == 0) {
    // after a timeout: copies of issued tokens k .. may still be landing
    for (int64_t j = k; j < n_my && j < k + kBgSlots; ++j)
      mbar_wait(smem_u32(bars + j % kBgSlots), static_cast<uint32_t>((j / kBgSlots) & 1), nullptr);
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Page-ordered walk (for tables in host memory). The GPU translates host
// addresses through a cache of limited reach: a random row gather over a
// 32 GB host table misses it on almost every row and runs at a tenth of the
// link rate, while the same rows read in table order run at the link rate
// (measured on a GB300: 16 vs 197 GB/s). The ordered gather first sorts the
// (token, head) items by the 2 MiB span of the table their row lies in
// (counting sort: count, scan, scatter), then walks them in that order and
// writes every row to its own output slot, so the result is identical.
// ---------------------------------------------------------------------------
constexpr int kOrderThreads = 256;
constexpr int kScanThreads = 1024;
constexpr uint32_t kMaxBuckets = 1u << 20;

struct OrderPlan {
  int shift;         // rows of one bucket = 2^shift (2 MiB of table, or more)
  uint32_t buckets;  // spans of the table + one bucket for ids outside it
  size_t counts_off, cursor_off, perm_off, bytes;
};

OrderPlan order_plan(int64_t items, int64_t table_rows, int row_bytes) {
  OrderPlan p{};
  int shift = 0;
  while ((static_cast<int64_t>(row_bytes) << (shift + 1)) <= (int64_t(2) << 20)) ++shift;
  while (((table_rows + (int64_t(1) << shift) - 1) >> shift) + 1 > kMaxBuckets) ++shift;
  p.shift = shift;
  p.buckets = static_cast<uint32_t>(((table_rows + (int64_t(1) << shift) - 1) >> shift) + 1);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  p.counts_off = 0;
  p.cursor_off = up(static_cast<size_t>(p.buckets) * 4);
  p.perm_off = p.cursor_off + up(static_cast<size_t>(p.buckets) * 4);
  p.bytes = p.perm_off + up(static_cast<size_t>(items) * 4);
  return p;
}

__device__ __forceinline__ uint32_t bucket_of(int64_t id, int64_t rows, int shift,
                                              uint32_t buckets) {
  return static_cast<uint64_t>(id) < static_cast<uint64_t>(rows)
             ? static_cast<uint32_t>(id >> shift)
             : buckets - 1;
}

__global__ void __launch_bounds__(kOrderThreads)
order_count_kernel(const int64_t* __restrict__ ids, uint32_t items, int64_t rows, int shift,
                   uint32_t buckets, uint32_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  for (uint32_t i = blockIdx.x * kOrderThreads + threadIdx.x; i < items;
       i += gridDim.x * kOrderThreads)
    atomicAdd(counts + bucket_of(__ldg(ids + i), rows, shift, buckets), 1u);
}

// Exclusive prefix sum of counts[0, n) into cursor[0, n), one CTA.
__global__ void __launch_bounds__(kScanThreads)
order_scan_kernel(const uint32_t* __restrict__ counts, uint32_t n, uint32_t* __restrict__ cursor) {
  __shared__ uint32_t warp_tot[kScanThreads / 32];
  pdl_wait();
  pdl_trigger();
  const uint32_t tid = threadIdx.x;
  const uint32_t chunk = (n + kScanThreads - 1) / kScanThreads;
  const uint32_t b0 = tid * chunk;
  const uint32_t b1 = min(b0 + chunk, n);
  uint32_t sum = 0;
  for (uint32_t b = b0; b < b1; ++b) sum += counts[b];
  // block-wide exclusive scan of the per-thread sums
  uint32_t x = sum;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  uint32_t run = x - sum + (warp > 0 ? warp_tot[warp - 1] : 0u);
  for (uint32_t b = b0; b < b1; ++b) {
    const uint32_t c = counts[b];
    cursor[b] = run;
    run += c;
  }
}

__global__ void __launch_bounds__(kOrderThreads)
order_scatter_kernel(const int64_t* __restrict__ ids, uint32_t items, int64_t rows, int shift,
                     uint32_t buckets, uint32_t* __restrict__ cursor,
                     uint32_t* __restrict__ perm) {
  pdl_wait();
  pdl_trigger();
  for (uint32_t i = blockIdx.x * kOrderThreads + threadIdx.x; i < items;
       i += gridDim.x * kOrderThreads) {
    const uint32_t b = bucket_of(__ldg(ids + i), rows, shift, buckets);
    perm[atomicAdd(cursor + b, 1u)] = i;
  }
}

// A validated gather: everything the kernels need.
struct Gather {
  const int64_t* ids;
  int64_t items;      // num_tokens * num_heads
  int64_t table_rows;
  int vpr;            // 16-byte vectors per table row
  int row_bytes;
  ple_dtype dtype;
  const float* row_scale;
  const uint4* table;  // device view
  uint4* out;
  uint32_t total_vecs;
  unsigned grid;
  int32_t* dev_err;
};

ple_status prepare_gather(const int64_t* ids, int64_t num_tokens, int32_t num_heads,
                          const void* table, int64_t table_rows, int32_t head_dim,
                          ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                          ple_bf16_t* out, int32_t max_ctas, int32_t* dev_err,
                          const char* name, Gather* g, bool* empty, bool ids_in = true) {
  *empty = false;
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1 || table_rows < 0)
    return fail(PLE_ERR_INVALID_ARG, "%s: bad sizes (T=%lld H=%d D=%d rows=%lld)", name,
                static_cast<long long>(num_tokens), num_heads, head_dim,
                static_cast<long long>(table_rows));
  if (dtype != PLE_BF16 && dtype != PLE_FP8_E4M3 && dtype != PLE_FP8_E4M3_TENSOR)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown dtype %d", name, static_cast<int>(dtype));
  if (loc != PLE_HBM && loc != PLE_HOST_UVA)
    return fail(PLE_ERR_INVALID_ARG, "%s: unknown table location %d", name, static_cast<int>(loc));
  const int elem = (dtype == PLE_BF16) ? 2 : 1;
  if ((static_cast<int64_t>(head_dim) * elem) % 16 != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: row of %d bytes is not a multiple of 16", name,
                head_dim * elem);
  if (num_tokens == 0) {
    *empty = true;
    return PLE_OK;
  }
  if ((ids_in && !ids) || !table || !out)
    return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (dtype != PLE_BF16 && !row_scale)
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
  int64_t blocks = (total + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int64_t full_grid = static_cast<int64_t>(num_sms()) * (2048 / kThreads);
  if (blocks > full_grid) blocks = full_grid;
  if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
  g->ids = ids;
  g->items = num_tokens * num_heads;
  g->table_rows = table_rows;
  g->vpr = vpr;
  g->row_bytes = vpr * 16;
  g->dtype = dtype;
  g->row_scale = row_scale;
  // Read the table through the device view of the allocation (identical to
  // the host address under unified addressing, but ask rather than assume).
  g->table = static_cast<const uint4*>(attr.devicePointer ? attr.devicePointer : table);
  g->out = reinterpret_cast<uint4*>(out);
  g->total_vecs = static_cast<uint32_t>(total);
  g->grid = static_cast<unsigned>(blocks < 1 ? 1 : blocks);
  g->dev_err = dev_err;
  return PLE_OK;
}

ple_status launch_gather_kernel(const Gather& g, const uint32_t* perm, cudaStream_t stream,
                                const char* name) {
  const int vpr = g.vpr;
  cudaError_t err = cudaSuccess;
  if (g.dtype == PLE_BF16) {
    if (vpr == 16)
      err = launch_kernel_pdl(perm == nullptr, gather_bf16_kernel<16>, dim3(g.grid), dim3(kThreads), 0, stream, 1, g.ids, perm, g.total_vecs, vpr, g.table, g.table_rows, g.out, g.dev_err);
    else if (vpr == 8)
      err = launch_kernel_pdl(perm == nullptr, gather_bf16_kernel<8>, dim3(g.grid), dim3(kThreads), 0, stream, 1, g.ids, perm, g.total_vecs, vpr, g.table, g.table_rows, g.out, g.dev_err);
    else
      err = launch_kernel_pdl(perm == nullptr, gather_bf16_kernel<0>, dim3(g.grid), dim3(kThreads), 0, stream, 1, g.ids, perm, g.total_vecs, vpr, g.table, g.table_rows, g.out, g.dev_err);
  } else {
    if (vpr == 8)
      err = launch_kernel_pdl(perm == nullptr, gather_fp8_kernel<8>, dim3(g.grid), dim3(kThreads), 0, stream, 1, g.ids, perm, g.total_vecs, vpr, g.table, g.row_scale, g.dtype == PLE_FP8_E4M3 ? 1 : 0, g.table_rows, g.out, g.dev_err);
    else
      err = launch_kernel_pdl(perm == nullptr, gather_fp8_kernel<0>, dim3(g.grid), dim3(kThreads), 0, stream, 1, g.ids, perm, g.total_vecs, vpr, g.table, g.row_scale, g.dtype == PLE_FP8_E4M3 ? 1 : 0, g.table_rows, g.out, g.dev_err);
  }
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}

ple_status launch_gather(const int64_t* ids, int64_t num_tokens, int32_t num_heads,
                         const void* table, int64_t table_rows, int32_t head_dim,
                         ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                         ple_bf16_t* out, int32_t max_ctas, int32_t* dev_err,
                         cudaStream_t stream, const char* name) {
  Gather g{};
  bool empty = false;
  ple_status s = prepare_gather(ids, num_tokens, num_heads, table, table_rows, head_dim, dtype,
                                row_scale, loc, out, max_ctas, dev_err, name, &g, &empty);
  if (s != PLE_OK || empty) return s;
  // PLE_GATHER_MODE=bulk sends bf16 rows in HBM through the copy engine when a
  // token's rows fit the slots (sweeps, tests); the register-fed kernel is the
  // default: on a GB300 at 8k prefill both take the same time.
  const size_t tok_bytes = static_cast<size_t>(num_heads) * g.row_bytes;
  const size_t smem = static_cast<size_t>(kBgWarps) * kBgSlots * (tok_bytes + 8);
  const char* mode = getenv("PLE_GATHER_MODE");
  const bool bulk = mode != nullptr && strcmp(mode, "bulk") == 0;
  if (bulk && dtype == PLE_BF16 && loc == PLE_HBM && smem <= kBgSmemBudget) {
    cudaError_t err = cudaFuncSetAttribute(gather_bulk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return check_cuda(err, name);
    // as many CTAs as fit (shared memory), at least one token per warp
    const int64_t per_sm = static_cast<int64_t>(kBgSmemBudget) / static_cast<int64_t>(smem);
    int64_t grid = static_cast<int64_t>(num_sms()) * (per_sm < 1 ? 1 : per_sm);
    const int64_t by_tokens = (num_tokens + kBgWarps - 1) / kBgWarps;
    if (grid > by_tokens) grid = by_tokens;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    if (grid < 1) grid = 1;
    err = launch_kernel(gather_bulk_kernel, dim3(static_cast<unsigned>(grid)), dim3(kBgWarps * 32),
                        smem, stream, 1, ids, num_tokens, static_cast<int>(num_heads),
                        g.row_bytes, reinterpret_cast<const uint8_t*>(g.table), table_rows,
                        reinterpret_cast<uint8_t*>(g.out), dev_err);
    if (err != cudaSuccess) return check_cuda(err, name);
    return check_cuda(cudaGetLastError(), name);
  }
  // Default: the token-major kernel when the shape fits it (PLE_GATHER_MODE=
  // vector keeps the vector-strided kernel: sweeps and tests).
  const int tpw = tok_group(num_heads, g.vpr);
  const bool vector_mode = mode != nullptr && strcmp(mode, "vector") == 0;
  if (tpw > 0 && !vector_mode && loc == PLE_HBM && (g.vpr == 8 || g.vpr == 16)) {
    const int64_t groups = (num_tokens + tpw - 1) / tpw;
    int64_t blocks = (groups + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t full = static_cast<int64_t>(num_sms()) * (dtype == PLE_BF16 ? 4 : 3);
    if (blocks > full) blocks = full;
    if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
    const dim3 grid(static_cast<unsigned>(blocks < 1 ? 1 : blocks));
    const int sstride = dtype == PLE_FP8_E4M3 ? 1 : 0;
    cudaError_t err;
    if (dtype == PLE_BF16)
      err = g.vpr == 16
                ? launch_kernel(gather_tok_kernel<16, false>, grid, dim3(kThreads), 0, stream, 1,
                                ids, num_tokens, static_cast<int>(num_heads), tpw, g.table,
                                row_scale, sstride, table_rows, g.out, dev_err)
                : launch_kernel(gather_tok_kernel<8, false>, grid, dim3(kThreads), 0, stream, 1,
                                ids, num_tokens, static_cast<int>(num_heads), tpw, g.table,
                                row_scale, sstride, table_rows, g.out, dev_err);
    else
      err = g.vpr == 16
                ? launch_kernel(gather_tok_kernel<16, true>, grid, dim3(kThreads), 0, stream, 1,
                                ids, num_tokens, static_cast<int>(num_heads), tpw, g.table,
                                row_scale, sstride, table_rows, g.out, dev_err)
                : launch_kernel(gather_tok_kernel<8, true>, grid, dim3(kThreads), 0, stream, 1,
                                ids, num_tokens, static_cast<int>(num_heads), tpw, g.table,
                                row_scale, sstride, table_rows, g.out, dev_err);
    if (err != cudaSuccess) return check_cuda(err, name);
    return check_cuda(cudaGetLastError(), name);
  }
  return launch_gather_kernel(g, nullptr, stream, name);
}

// Sort the items by table span into the workspace, then gather in that order.
ple_status launch_ordered(const Gather& g, uint8_t* ws, const OrderPlan& plan,
                          cudaStream_t stream, const char* name) {
  uint32_t* counts = reinterpret_cast<uint32_t*>(ws + plan.counts_off);
  uint32_t* cursor = reinterpret_cast<uint32_t*>(ws + plan.cursor_off);
  uint32_t* perm = reinterpret_cast<uint32_t*>(ws + plan.perm_off);
  const uint32_t items = static_cast<uint32_t>(g.items);
  cudaError_t err = cudaMemsetAsync(counts, 0, static_cast<size_t>(plan.buckets) * 4, stream);
  if (err != cudaSuccess) return check_cuda(err, name);
  int64_t blocks = (g.items + kOrderThreads - 1) / kOrderThreads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 4;
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  // plain stream order for the sort (see the walk's note on early launches)
  err = launch_kernel_pdl(false, order_count_kernel, dim3(grid), dim3(kOrderThreads), 0, stream,
                          1, g.ids, items, g.table_rows, plan.shift, plan.buckets, counts);
  if (err == cudaSuccess)
    err = launch_kernel_pdl(false, order_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, 1,
                            static_cast<const uint32_t*>(counts), plan.buckets, cursor);
  if (err == cudaSuccess)
    err = launch_kernel_pdl(false, order_scatter_kernel, dim3(grid), dim3(kOrderThreads), 0,
                            stream, 1, g.ids, items, g.table_rows, plan.shift, plan.buckets,
                            cursor, perm);
  if (err != cudaSuccess) return check_cuda(err, name);
  ple_status s = check_cuda(cudaGetLastError(), name);
  if (s != PLE_OK) return s;
  // Two CTAs per SM walk the sorted items: a slice of ~2.5 MB of rows in
  // flight, enough for the host link, narrow enough to stay within the
  // GPU's translation reach (a full grid spreads its rows over half the table).
  Gather gw = g;
  const unsigned walk_ctas = static_cast<unsigned>(2 * num_sms());
  if (gw.grid > walk_ctas) gw.grid = walk_ctas;
  return launch_gather_kernel(gw, perm, stream, name);
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

PLE_EXPORT size_t ple_lookup_ordered_workspace(int64_t num_tokens, int32_t num_heads,
                                               int64_t table_rows, int32_t head_dim,
                                               ple_dtype dtype) {
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1 || table_rows < 0) return 0;
  if (dtype != PLE_BF16 && dtype != PLE_FP8_E4M3 && dtype != PLE_FP8_E4M3_TENSOR) return 0;
  const int elem = (dtype == PLE_BF16) ? 2 : 1;
  const int row_bytes = static_cast<int>((static_cast<int64_t>(head_dim) * elem + 15) / 16 * 16);
  return ple::order_plan(num_tokens * num_heads, table_rows, row_bytes).bytes;
}

PLE_EXPORT ple_status ple_lookup_ordered(const int64_t* ids, int64_t num_tokens,
                                         int32_t num_heads, const void* table,
                                         int64_t table_rows, int32_t head_dim, ple_dtype dtype,
                                         const float* row_scale, ple_table_loc loc,
                                         ple_bf16_t* out, int32_t max_ctas, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err,
                                         cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_lookup_ordered";
  Gather g{};
  bool empty = false;
  ple_status s = prepare_gather(ids, num_tokens, num_heads, table, table_rows, head_dim, dtype,
                                row_scale, loc, out, max_ctas, dev_err, name, &g, &empty);
  if (s != PLE_OK || empty) return s;
  const OrderPlan plan = order_plan(g.items, table_rows, g.row_bytes);
  if (workspace == nullptr || workspace_bytes < plan.bytes)
    return fail(PLE_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name,
                workspace_bytes, plan.bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PLE_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", name);
  return launch_ordered(g, static_cast<uint8_t*>(workspace), plan, stream, name);
}

// ---------------------------------------------------------------------------
// ple_lookup_ordered_static: ple_lookup_ordered without a caller workspace.
// For callers that may not allocate device memory on their serving path: an
// engine that carves all device memory into its own pools at start-up and
// forbids any later allocation, or a C caller with no device allocator of
// its own. The sort's scratch (bucket counters, cursors, walk order) lives in
// one file-scope device array of fixed size per device instead; the call
// allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
// ---------------------------------------------------------------------------
namespace ple {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) uint8_t g_order_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<uint8_t*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (cudaGetSymbolAddress) and cached.
ple_status static_scratch(uint8_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return check_cuda(err, "ple_lookup_ordered_static: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(PLE_ERR_UNSUPPORTED, "ple_lookup_ordered_static: device %d beyond %d", dev,
                kMaxDevices);
  uint8_t* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* sym = nullptr;
    err = cudaGetSymbolAddress(&sym, g_order_scratch);
    if (err != cudaSuccess)
      return check_cuda(err, "ple_lookup_ordered_static: cudaGetSymbolAddress");
    p = static_cast<uint8_t*>(sym);
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PLE_OK;
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_lookup_ordered_static(const int64_t* ids, int64_t num_tokens,
                                                int32_t num_heads, const void* table,
                                                int64_t table_rows, int32_t head_dim,
                                                ple_dtype dtype, const float* row_scale,
                                                ple_table_loc loc, ple_bf16_t* out,
                                                int32_t max_ctas, int32_t* dev_err,
                                                cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_lookup_ordered_static";
  Gather g{};
  bool empty = false;
  ple_status s = prepare_gather(ids, num_tokens, num_heads, table, table_rows, head_dim, dtype,
                                row_scale, loc, out, max_ctas, dev_err, name, &g, &empty);
  if (s != PLE_OK || empty) return s;
  const OrderPlan plan = order_plan(g.items, table_rows, g.row_bytes);
  if (plan.bytes > kStaticScratchBytes)
    return fail(PLE_ERR_UNSUPPORTED,
                "%s: %lld items over %lld table rows need %zu bytes of scratch, above the "
                "%zu-byte static scratch (use ple_lookup_ordered with a workspace)",
                name, static_cast<long long>(g.items), static_cast<long long>(table_rows),
                plan.bytes, kStaticScratchBytes);
  uint8_t* scratch = nullptr;
  s = static_scratch(&scratch);
  if (s != PLE_OK) return s;
  return launch_ordered(g, scratch, plan, stream, name);
}

PLE_EXPORT ple_status ple_ngram_lookup(const int32_t* input_ids, int64_t num_tokens,
                                       const int32_t* query_start_loc, int32_t num_reqs,
                                       const int32_t* ngram_context, int32_t ctx_len,
                                       const int64_t* layer_multipliers,
                                       const int64_t* vocab_sizes, const int64_t* offsets,
                                       int32_t eos_token_id, int32_t heads_per_ngram,
                                       const void* table, int64_t table_rows, int32_t head_dim,
                                       ple_dtype dtype, const float* row_scale, ple_table_loc loc,
                                       ple_bf16_t* out, int64_t* ids_out,
                                       int32_t* ngram_context_out, int32_t max_ctas,
                                       int32_t* dev_err, cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_ngram_lookup";
  if (num_tokens < 0) return fail(PLE_ERR_INVALID_ARG, "%s: num_tokens < 0", name);
  NgramConsts k{};
  int num_heads = 0;
  ple_status s = make_ngram_consts(ctx_len, heads_per_ngram, layer_multipliers, vocab_sizes,
                                   offsets, &k, &num_heads, name);
  if (s != PLE_OK) return s;
  if (num_reqs < 0 || (num_reqs == 0 && num_tokens > 0))
    return fail(PLE_ERR_INVALID_ARG, "%s: num_reqs must be >= 1 when there are tokens", name);
  for (int h = 0; h < num_heads; ++h)
    if (offsets[h] < 0 || offsets[h] > table_rows - vocab_sizes[h])
      return fail(PLE_ERR_INVALID_ARG, "%s: head %d's partition [%lld, %lld + %lld) is outside "
                  "the table's %lld rows", name, h, static_cast<long long>(offsets[h]),
                  static_cast<long long>(offsets[h]), static_cast<long long>(vocab_sizes[h]),
                  static_cast<long long>(table_rows));
  if (ngram_context_out && ngram_context &&
      overlaps(ngram_context, sizeof(int32_t) * num_reqs * ctx_len, ngram_context_out,
               sizeof(int32_t) * num_reqs * ctx_len))
    return fail(PLE_ERR_INVALID_ARG, "%s: ngram_context_out overlaps ngram_context", name);
  Gather g;
  bool empty = false;
  s = prepare_gather(ids_out, num_tokens, num_heads, table, table_rows, head_dim, dtype,
                     row_scale, loc, out, max_ctas, dev_err, name, &g, &empty,
                     /*ids_in=*/false);
  if (s != PLE_OK) return s;
  if (empty) {
    // no tokens: the carry-over is the history itself (EOS without one)
    if (ngram_context_out == nullptr || num_reqs == 0) return PLE_OK;
    if (ngram_context != nullptr)
      return copy_carry(ngram_context_out, ngram_context, sizeof(int32_t) * num_reqs * ctx_len,
                        stream);
    return ple_ngram_ids(input_ids, 0, query_start_loc, num_reqs, nullptr, ctx_len,
                         layer_multipliers, vocab_sizes, offsets, eos_token_id, heads_per_ngram,
                         nullptr, ngram_context_out, dev_err, stream);
  }
  if (!input_ids || !query_start_loc)
    return fail(PLE_ERR_INVALID_ARG, "%s: null device pointer", name);
  NgramArgs na{};
  na.input_ids = input_ids;
  na.num_tokens = num_tokens;
  na.qsl = query_start_loc;
  na.num_reqs = num_reqs;
  na.ctx = ngram_context;
  na.ctx_len = ctx_len;
  na.eos = eos_token_id;
  na.heads_per_ngram = heads_per_ngram;
  na.num_heads = num_heads;
  na.ctx_out = ngram_context_out;
  na.ids_out = ids_out;
  const int scale_stride = dtype == PLE_FP8_E4M3 ? 1 : 0;
  cudaError_t err;
  // Token-major kernel where the shape fits it (PLE_GATHER_MODE=vector keeps
  // the vector-strided one: sweeps and tests).
  const int tpw = tok_group(num_heads, g.vpr);
  const char* mode = getenv("PLE_GATHER_MODE");
  const bool vector_mode = mode != nullptr && strcmp(mode, "vector") == 0;
  if (tpw > 0 && !vector_mode && (g.vpr == 8 || g.vpr == 16)) {
    const int64_t groups = (num_tokens + tpw - 1) / tpw;
    int64_t blocks = (groups + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t full = static_cast<int64_t>(num_sms()) * (dtype == PLE_BF16 ? 4 : 3);
    if (blocks > full) blocks = full;
    if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
    const dim3 grid(static_cast<unsigned>(blocks < 1 ? 1 : blocks));
    if (dtype == PLE_BF16)
      err = g.vpr == 16 ? launch_kernel(ngram_tok_kernel<16, false>, grid, dim3(kThreads), 0,
                                        stream, 1, na, k, tpw, g.table, g.row_scale, 0,
                                        g.table_rows, g.out, dev_err)
                        : launch_kernel(ngram_tok_kernel<8, false>, grid, dim3(kThreads), 0,
                                        stream, 1, na, k, tpw, g.table, g.row_scale, 0,
                                        g.table_rows, g.out, dev_err);
    else
      err = g.vpr == 16 ? launch_kernel(ngram_tok_kernel<16, true>, grid, dim3(kThreads), 0,
                                        stream, 1, na, k, tpw, g.table, g.row_scale,
                                        scale_stride, g.table_rows, g.out, dev_err)
                        : launch_kernel(ngram_tok_kernel<8, true>, grid, dim3(kThreads), 0,
                                        stream, 1, na, k, tpw, g.table, g.row_scale,
                                        scale_stride, g.table_rows, g.out, dev_err);
    if (err != cudaSuccess) return check_cuda(err, name);
    return check_cuda(cudaGetLastError(), name);
  }
  if (dtype == PLE_BF16) {
    err = g.vpr == 16
              ? launch_kernel(ngram_gather_kernel<16, false>, dim3(g.grid), dim3(kThreads), 0,
                              stream, 1, na, k, g.total_vecs, g.vpr, g.table, g.row_scale, 0,
                              g.table_rows, g.out, dev_err)
              : launch_kernel(ngram_gather_kernel<0, false>, dim3(g.grid), dim3(kThreads), 0,
                              stream, 1, na, k, g.total_vecs, g.vpr, g.table, g.row_scale, 0,
                              g.table_rows, g.out, dev_err);
  } else {
    err = g.vpr == 8
              ? launch_kernel(ngram_gather_kernel<8, true>, dim3(g.grid), dim3(kThreads), 0,
                              stream, 1, na, k, g.total_vecs, g.vpr, g.table, g.row_scale,
                              scale_stride, g.table_rows, g.out, dev_err)
              : launch_kernel(ngram_gather_kernel<0, true>, dim3(g.grid), dim3(kThreads), 0,
                              stream, 1, na, k, g.total_vecs, g.vpr, g.table, g.row_scale,
                              scale_stride, g.table_rows, g.out, dev_err);
  }
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}
