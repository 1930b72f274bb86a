// ple_kv_proj / ple_kv_proj_gate: the merged key/value projection
// kv = emb @ W^T on the 5th-generation tensor cores (tcgen05.mma,
// accumulators in tensor memory), operands staged by TMA; ple_kv_proj_gate
// also reduces the gate's row sums from the key tiles in the epilogue.
//
// Source: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), 实现拆解 item 1:
// key_proj and value_proj merged into one MergedColumnParallelLinear, so one
// GEMM [T, E] x [2C, E]^T produces k (columns [0, C)) and v ([C, 2C)).
//
// Two kernels: the CTA-pair kernel further below (the default: cta_group::2
// MMAs over 256 x 256 tiles) and the one-SM kernel described here (for at
// most 128 rows, and the launch-shape variants). Design of the one-SM kernel
// (dense contraction, tensor-bound at serving sizes):
//   * CTA tile 128 x 256 (M x N), K step 64 = one 128-byte swizzle atom of
//     bf16. A = emb and B = W are both K-major, exactly the canonical
//     SWIZZLE_128B K-major layout TMA writes and tcgen05 reads, so no
//     transposes anywhere. tcgen05.mma.cta_group::1.kind::f16, M=128 N=256
//     K=16, fp32 accumulate.
//   * 4-stage smem ring (48 KB per stage) fed by TMA; mbarriers full/empty.
//   * Persistent: one CTA per SM walks tiles tile = blockIdx.x + i*gridDim.x
//     (consecutive CTAs share A rows; all of W stays hot in the 129 MB L2).
//   * Two 256-column fp32 accumulators in TMEM (all 512 columns): the
//     epilogue of tile i drains one while the MMAs of tile i+1 fill the other.
//   * Warp roles (192 threads): warp 0 lane 0 issues TMA, warp 1 owns TMEM and
//     lane 0 issues MMAs, warps 2-5 (one per TMEM lane quadrant) read the
//     accumulator with tcgen05.ld, round to bf16 and store rows to global.
//   * Every mbarrier wait is bounded (1 s of %globaltimer). On expiry the
//     kernel raises PLE_DEVERR_TIMEOUT, stops issuing, waits (bounded) for its
//     own TMA copies and MMAs in flight, frees TMEM and returns.
#include "common.cuh"
#include "tma.cuh"

#include <cstdlib>
#include <cstring>

namespace ple {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int A_STAGE = BM * BK * 2;     // 16 KB
constexpr int B_STAGE = BN * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int ACC_COLS = BN;             // fp32 columns per accumulator
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr int kNumBars = 2 * STAGES + 4 + 1;
constexpr size_t kSmemBytes = size_t(STAGES) * STAGE_BYTES + 1024 /*align*/ + 256 /*bars*/;

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), A and B K-major (15, 16 = 0), N >> 3 at 17-22,
// M >> 4 at 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// tile whose rows are 128 bytes and whose 8-row groups are 1024 bytes apart:
// start address >> 4 (bits 0-13), leading byte offset (16-29; not used by
// swizzled K-major layouts, set to 1), stride byte offset 1024 >> 4 (32-45),
// fixed 0b001 at 46-48, base offset 0 (tiles are 1024-byte aligned),
// swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      // the wait sits in the same statement so no use of r[] can move above it
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(lo_f32), __uint_as_float(hi_f32));
  return *reinterpret_cast<const uint32_t*>(&b);
}

// One CTA per 128 x 256 tile (the kernel for at most 128 rows; the pair
// kernel below takes everything larger).
__global__ void __launch_bounds__(kThreads, 1)
kv_proj_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               ple_bf16_t* __restrict__ out, int M, int N, int K, int32_t* dev_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* a_smem = smem;
  uint8_t* b_smem = smem + STAGES * A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cluster_id = blockIdx.x;
  const int num_clusters = gridDim.x;
  const int n_tiles = (N + BN - 1) / BN;
  const int num_tiles = ((M + BM - 1) / BM) * n_tiles;
  const int num_kb = (K + BK - 1) / BK;
  // tile -> (m block, n block)
  auto m_block = [&](int tile) { return tile / n_tiles; };
  auto n_block = [&](int tile) { return tile % n_tiles; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // released by the MMAs' commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpilogueThreads);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // emb (A) comes from the previous kernel
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0;        // stages holding a copy this thread issued
    uint32_t armed_parity = 0; // parity of that copy's full-barrier phase
    bool ok = true;
    for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
      const int m0 = m_block(tile) * BM;
      const int n0 = n_block(tile) * BN;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
        tma_load_2d(smem_u32(a_smem + stage * A_STAGE), &map_a, full_bar(stage), kb * BK, m0);
        tma_load_2d(smem_u32(b_smem + stage * B_STAGE), &map_b, full_bar(stage), kb * BK, n0);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
    // Never leave with a copy in flight into this CTA's shared memory.
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u, nullptr);
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a_desc = sw128_desc(smem_u32(a_smem + stage * A_STAGE));
          const uint64_t b_desc = sw128_desc(smem_u32(b_smem + stage * B_STAGE));
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // advance 16 elements (32 bytes) along K inside the swizzle atom
            const uint64_t koff = static_cast<uint64_t>((kk * UMMA_K * 2) >> 4);
            umma_bf16(d_tmem, a_desc + koff, b_desc + koff, (kb | kk) != 0 ? 1u : 0u);
          }
          // frees the stage once these MMAs finish
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(accf_bar(acc));        // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
      // Every MMA this thread issued has completed once done_bar flips.
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> registers -> bf16 -> global ----------------
    const int quad = warp & 3;                 // TMEM lanes this warp may read
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster_id; tile < num_tiles; tile += num_clusters) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(accf_bar(acc), acc_phase, abort_flag));
      if (!ok) {
        if (lane == 0) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
        break;
      }
      tc_fence_after();
      const int m = m_block(tile) * BM + row_in_tile;
      const int n_base = n_block(tile) * BN;
      ple_bf16_t* row_out = out + static_cast<int64_t>(m) * N;
#pragma unroll 1
      for (int chunk = 0; chunk < BN / 32; ++chunk) {
        uint32_t r[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                      static_cast<uint32_t>(acc * ACC_COLS + chunk * 32),
                  r);
        const int n = n_base + chunk * 32;
        if (m < M && n < N) {
          uint4* dst = reinterpret_cast<uint4*>(row_out + n);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(r[8 * q + 0], r[8 * q + 1]);
            v.y = pack_bf16x2(r[8 * q + 2], r[8 * q + 3]);
            v.z = pack_bf16x2(r[8 * q + 4], r[8 * q + 5]);
            v.w = pack_bf16x2(r[8 * q + 6], r[8 * q + 7]);
            dst[q] = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acce_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel: tcgen05.mma.cta_group::2, M = 256 (128 rows per SM) x
// N = 256 (128, 192 or 64 for the narrower units of pair_unit's schedules).
// Each CTA of a cluster pair stages its own 128 rows of A and its own
// half (128 rows) of the W tile; the pair's tensor cores read both halves of
// W, so each SM reads 32 KB of operands from shared memory per K step of 64
// instead of 48 KB. The even CTA (leader) issues the MMAs; TMA copies of both CTAs
// complete on the leader's full barrier; the leader's commits release the
// stages and hand the accumulators to the epilogues of both CTAs; both
// epilogues report back to the leader's accumulator-empty barrier.
// ---------------------------------------------------------------------------
// A stage holds two 64-wide K atoms (128 of K) of both operands: 3 stages of
// 64 KB per CTA. Measured on a GB300 at 8192 x 2048 -> 8192: 153 us against
// 169 us for 7 stages of one atom (half the full/empty handshakes per MMA)
// and 172 us for 2 stages of three.
constexpr int P_STAGES = 3;
constexpr int P_ATOMS = 2;                      // 64-wide K atoms per stage
constexpr int P_A_ATOM = BM * BK * 2;           // 16 KB
constexpr int P_B_ATOM = (BN / 2) * BK * 2;     // 16 KB
constexpr int P_A_STAGE = P_ATOMS * P_A_ATOM;
constexpr int P_B_STAGE = P_ATOMS * P_B_ATOM;
constexpr int P_STAGE_BYTES = P_A_STAGE + P_B_STAGE;
constexpr int P_NUM_BARS = 2 * P_STAGES + 4 + 1;
constexpr size_t kPairSmemBytes = size_t(P_STAGES) * P_STAGE_BYTES + 1024 + 256;
// Epilogue warps: 4 (one per TMEM lane quadrant, each draining all columns
// of a unit) or 8 (two per quadrant, each draining one half of them).
// With few tiles per CTA the last tile's epilogue, which nothing hides, is a
// large share of the launch and 8 warps halve it (29.5 against 30.7 us for
// 1024 x 2048 -> 8192 with the fused gate on a GB300); with many tiles the
// epilogues are hidden behind the MMAs and the extra warps only compete
// with the issuing warps (1 % slower at 32768 rows).
template <int EW>
constexpr int pair_threads() { return 64 + 32 * EW; }
constexpr int kFewRounds = 4;  // at most this many tiles per CTA pair: 8 epilogue warps
constexpr size_t kKeyFirstMaxA = size_t(64) << 20;  // bytes of A for the key-first order
// kind::f16 instruction descriptor for M = 256 (two SMs) x N = cols (a
// multiple of 16 up to 256: the full, half and value-strip tiles): D f32, A
// and B bf16, both K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_pair(int cols) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(cols >> 3) << 17) |
         (uint32_t((2 * BM) >> 4) << 24);
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at offset `bar` in every CTA of ctaMask once the
// pair MMAs issued so far complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// Fused gate reductions (ple_kv_proj_gate). The key half of kv is never
// stored: the epilogue of a key tile (columns [n, n+256) or, for a half
// tile, [n, n+128) of [0, C)) rounds each accumulator to bf16 -- the value
// ple_kv_proj would store -- reads the same channels of the token's hidden
// row and adds, per row and 128-channel block, sum h^2, sum k^2 and
// sum h*k*gamma_h*gamma_k (the three sums of the gate's RMSNorm-and-dot,
// which split over channel blocks). Each block's triple goes to
// partial[block][row] -- the same sums in the same order whether the block
// came from a full or a half tile; the epilogue warp that delivers the last
// blocks of its 32 rows (a per-32-row arrival counter) adds the C/128 triples
// in block order, writes g = sigmoid(...) for those rows and sets the
// counter back to zero, so a launch that completes leaves every counter as
// it found it (zero) and the next launch needs no clearing pass. Value tiles
// are stored as in ple_kv_proj.
constexpr int kGateBlock = 128;  // channels per partial-sum block

struct GateEpi {
  const ple_bf16_t* hidden;   // [M][C]
  const ple_bf16_t* gamma_h;  // [C]
  const ple_bf16_t* gamma_k;  // [C]
  float4* partial;            // [C/128][M]: (sum h^2, sum k^2, sum h*k*gh*gk, 0)
  unsigned* count_top;        // one past the arrival counters: group j (rows 32j..32j+31)
                              // counts at count_top[-1 - j]; zero between launches
  float* gate_out;            // [M]
  float eps;
  int C;
};

__device__ __forceinline__ void gate_publish(const GateEpi& ge, int m, int M, int lane, int blk0,
                                             int nb, float4 part0, float4 part1);

// One key tile (cols = 256 or 128 channels from n_base) of the fused gate
// epilogue for this thread's row m (one warp = 32 consecutive rows). taddr:
// the warp's lane quadrant of the accumulator. Releases the accumulator to
// the MMA issuer (acce_bar of the pair leader) as soon as it is read, then
// publishes the row sums and, in the warp that completes its 32 rows, the
// gate scalars.
__device__ __forceinline__ void gate_tile(const GateEpi& ge, uint32_t taddr, int m, int M,
                                          int n_base, int cols, int lane, uint32_t leader,
                                          uint32_t acce_bar) {
  const bool row_ok = m < M;
  const ple_bf16_t* hrow = ge.hidden + static_cast<int64_t>(row_ok ? m : 0) * ge.C + n_base;
  const int n_chunks = cols / 32;
  uint64_t sh2 = 0, sk2 = 0, sd2 = 0;  // (+0.0f, +0.0f) pairs
  float4 part0 = make_float4(0.f, 0.f, 0.f, 0.f), part1 = part0;
  // h of the next chunk is in flight while this chunk is reduced
  uint4 hn[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) hn[q] = row_ok ? ldg16(hrow + q * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int c0 = chunk * 32;
    uint4 hv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hv[q] = hn[q];
      hn[q] = row_ok && chunk + 1 < n_chunks ? ldg16(hrow + c0 + 32 + q * 8)
                                             : make_uint4(0, 0, 0, 0);
    }
    uint32_t r[32];
    tmem_ld32(taddr + static_cast<uint32_t>(c0), r);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 ga = ldg16(ge.gamma_h + n_base + c0 + q * 8);  // warp-uniform
      const uint4 gb = ldg16(ge.gamma_k + n_base + c0 + q * 8);
      const uint32_t hw[4] = {hv[q].x, hv[q].y, hv[q].z, hv[q].w};
      const uint32_t aw[4] = {ga.x, ga.y, ga.z, ga.w};
      const uint32_t bw[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t kb = pack_bf16x2(r[8 * q + 2 * p], r[8 * q + 2 * p + 1]);
        const uint64_t k2 = f2(bf_lo(kb), bf_hi(kb));
        const uint64_t h2 = f2(bf_lo(hw[p]), bf_hi(hw[p]));
        const uint64_t gg = f2_mul(f2(bf_lo(aw[p]), bf_hi(aw[p])), f2(bf_lo(bw[p]), bf_hi(bw[p])));
        sh2 = f2_fma(h2, h2, sh2);
        sk2 = f2_fma(k2, k2, sk2);
        sd2 = f2_fma(f2_mul(h2, k2), gg, sd2);
      }
    }
    if ((chunk & 3) == 3) {  // a 128-channel block is complete
      float a0, a1, b0, b1, d0, d1;
      f2_split(sh2, a0, a1);
      f2_split(sk2, b0, b1);
      f2_split(sd2, d0, d1);
      const float4 pb = make_float4(a0 + a1, b0 + b1, d0 + d1, 0.f);
      if (chunk == 3) part0 = pb; else part1 = pb;
      sh2 = sk2 = sd2 = 0;
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar, leader));
  gate_publish(ge, m, M, lane, n_base / kGateBlock, cols / kGateBlock, part0, part1);
}

// Publishes a warp's block sums (nb = 1 or 2 blocks from blk0) for its rows
// and, in the warp that delivers the last block of its 32 rows, writes
// their gate scalars.
__device__ __forceinline__ void gate_publish(const GateEpi& ge, int m, int M, int lane, int blk0,
                                             int nb, float4 part0, float4 part1) {
  const bool row_ok = m < M;
  const int n_blk = ge.C / kGateBlock;
  if (row_ok) {
    ge.partial[static_cast<int64_t>(blk0) * M + m] = part0;
    if (nb == 2) ge.partial[static_cast<int64_t>(blk0 + 1) * M + m] = part1;
  }
  const int m0 = m - lane;  // first row of the warp
  if (m0 >= M) return;      // no row of this warp exists: nothing to count
  __threadfence();          // this lane's partials are visible GPU-wide ...
  __syncwarp();             // ... before lane 0 counts the warp's delivery
  unsigned* counter = ge.count_top - 1 - (m0 >> 5);
  unsigned last = 0;
  if (lane == 0)
    last = atomicAdd(counter, static_cast<unsigned>(nb)) + static_cast<unsigned>(nb) ==
           static_cast<unsigned>(n_blk);
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  if (lane == 0) *counter = 0;  // every arrival of this launch is in: ready for the next
  __threadfence();  // every other warp's partials of these rows are visible
  if (!row_ok) return;
  float sh = 0.f, sk = 0.f, sd = 0.f;
  for (int j = 0; j < n_blk; ++j) {
    const float4 p = __ldcg(ge.partial + static_cast<int64_t>(j) * M + m);
    sh += p.x;
    sk += p.y;
    sd += p.z;
  }
  ge.gate_out[m] = gate_of(sh, sk, sd, ge.C, ge.eps);
}

// The 8-warp epilogue's key block (128 channels from n_base, one per warp):
// all of the row's h and the block's gammas are loaded before the block's
// accumulator is ready (behind the MMAs), so the reduction waits on tensor
// memory alone. Lane l < 16 holds gamma_h of channels n_base + 8l .. + 7 and
// lane 16 + l gamma_k of the same channels; the chunks take them by shuffle.
struct GateBlockIn {
  uint4 h[kGateBlock / 32][4];
  uint4 gam;
};

__device__ __forceinline__ void gate_block_load(const GateEpi& ge, int m, int M, int n_base,
                                                int lane, GateBlockIn& in) {
  const bool row_ok = m < M;
  const ple_bf16_t* hrow = ge.hidden + static_cast<int64_t>(row_ok ? m : 0) * ge.C + n_base;
#pragma unroll
  for (int c = 0; c < kGateBlock / 32; ++c)
#pragma unroll
    for (int q = 0; q < 4; ++q)
      in.h[c][q] = row_ok ? ldg16(hrow + c * 32 + q * 8) : make_uint4(0, 0, 0, 0);
  in.gam = ldg16((lane < 16 ? ge.gamma_h : ge.gamma_k) + n_base + 8 * (lane & 15));
}

// The same sums, in the same order, as gate_tile over one block.
__device__ __forceinline__ void gate_block(const GateEpi& ge, uint32_t taddr, int m, int M,
                                           int n_base, int lane, uint32_t leader,
                                           uint32_t acce_bar, const GateBlockIn& in) {
  uint64_t sh2 = 0, sk2 = 0, sd2 = 0;  // (+0.0f, +0.0f) pairs
#pragma unroll
  for (int chunk = 0; chunk < kGateBlock / 32; ++chunk) {
    uint32_t r[32];
    tmem_ld32(taddr + static_cast<uint32_t>(chunk * 32), r);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int src = chunk * 4 + q;  // the lane holding these 8 channels' gamma_h
      const uint32_t aw[4] = {__shfl_sync(0xffffffffu, in.gam.x, src),
                              __shfl_sync(0xffffffffu, in.gam.y, src),
                              __shfl_sync(0xffffffffu, in.gam.z, src),
                              __shfl_sync(0xffffffffu, in.gam.w, src)};
      const uint32_t bw[4] = {__shfl_sync(0xffffffffu, in.gam.x, src + 16),
                              __shfl_sync(0xffffffffu, in.gam.y, src + 16),
                              __shfl_sync(0xffffffffu, in.gam.z, src + 16),
                              __shfl_sync(0xffffffffu, in.gam.w, src + 16)};
      const uint32_t hw[4] = {in.h[chunk][q].x, in.h[chunk][q].y, in.h[chunk][q].z,
                              in.h[chunk][q].w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t kb = pack_bf16x2(r[8 * q + 2 * p], r[8 * q + 2 * p + 1]);
        const uint64_t k2 = f2(bf_lo(kb), bf_hi(kb));
        const uint64_t h2 = f2(bf_lo(hw[p]), bf_hi(hw[p]));
        const uint64_t gg = f2_mul(f2(bf_lo(aw[p]), bf_hi(aw[p])), f2(bf_lo(bw[p]), bf_hi(bw[p])));
        sh2 = f2_fma(h2, h2, sh2);
        sk2 = f2_fma(k2, k2, sk2);
        sd2 = f2_fma(f2_mul(h2, k2), gg, sd2);
      }
    }
  }
  float a0, a1, b0, b1, d0, d1;
  f2_split(sh2, a0, a1);
  f2_split(sk2, b0, b1);
  f2_split(sd2, d0, d1);
  const float4 part = make_float4(a0 + a1, b0 + b1, d0 + d1, 0.f);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar, leader));
  gate_publish(ge, m, M, lane, n_base / kGateBlock, 1, part, part);
}

// A work unit of the pair kernel: 256 rows from m_base, `cols` columns from
// n_base. Default schedule: 256 x 256 tiles, and -- units >= full_units --
// 128-column halves of the last round's tiles (they let twice as many CTA
// pairs share that round when it would otherwise leave more than half of
// them idle). Strip schedule (vn > 0, the fused gate with key tiles first):
// the value half in strips of vn columns, the narrower strips left over at
// the end of each row block's value half (rem columns) first, then every key
// tile, then the vn-column strips: with units dealt to the pairs in turn, the
// host picks vn so that no pair gets much more than its share of columns
// (1024 x 2048 -> 8192 on 74 pairs: at most 1.75 tiles' columns per pair
// with vn = 192, against 2 tiles with 256-column tiles).
struct PairUnit {
  int m_base;
  int n_base;
  int cols;  // 256, 128, vn or rem
};

struct PairSched {
  int full_units;  // default schedule: units past it are half tiles
  int key_groups;  // > 0: key tiles first (C / 256 key groups)
  int vn;          // > 0: strip schedule
  int rem;         // strip schedule: columns left over per row block (0: none)
  int num_units;
};

// Tile v of the launch's tile order -> its 256-row block mb and 256-column
// group g. The natural order walks each row block's column groups in turn
// (consecutive CTA pairs share A rows). With key_groups > 0 (the fused gate's
// C / 256 key groups; used when each CTA pair has few tiles) every key tile
// comes first and every value tile after: the last round then holds value
// tiles, whose epilogue is a plain store, and the gate's completion of each
// row group runs behind the value tiles' MMAs instead of after them.
__device__ __forceinline__ void tile_of(int v, int n_groups, int key_groups, int m_tiles, int& mb,
                                        int& g) {
  if (key_groups == 0) {
    mb = v / n_groups;
    g = v % n_groups;
    return;
  }
  const int n_key = m_tiles * key_groups;
  if (v < n_key) {
    mb = v / key_groups;
    g = v % key_groups;
  } else {
    const int value_groups = n_groups - key_groups;
    mb = (v - n_key) / value_groups;
    g = key_groups + (v - n_key) % value_groups;
  }
}

// STRIPS: the kernel can run the strip schedule (the 8-warp kernels only:
// the host uses it for launches of few tiles per pair).
template <bool STRIPS>
__device__ __forceinline__ PairUnit pair_unit(int u, const PairSched& sc, int n_groups,
                                              int m_tiles) {
  PairUnit t;
  if (STRIPS && sc.vn > 0) {
    const int C = sc.key_groups * BN;
    const int strips = (C - sc.rem) / sc.vn;  // full strips per row block
    const int n_rem = sc.rem > 0 ? m_tiles : 0;
    const int n_key = m_tiles * sc.key_groups;
    int mb;
    if (u < n_rem) {
      mb = u;
      t.n_base = C + strips * sc.vn;
      t.cols = sc.rem;
    } else if (u - n_rem < n_key) {
      const int v = u - n_rem;
      mb = v / sc.key_groups;
      t.n_base = (v % sc.key_groups) * BN;
      t.cols = BN;
    } else {
      const int v = u - n_rem - n_key;
      mb = v / strips;
      t.n_base = C + (v % strips) * sc.vn;
      t.cols = sc.vn;
    }
    t.m_base = mb * 2 * BM;
    return t;
  }
  const int full_units = sc.full_units;
  const int key_groups = sc.key_groups;
  const int h = u - full_units;
  const int v = u >= full_units ? full_units + (h >> 1) : u;
  int mb, g;
  tile_of(v, n_groups, key_groups, m_tiles, mb, g);
  t.m_base = mb * 2 * BM;
  if (u >= full_units) {
    t.n_base = g * BN + (h & 1) * (BN / 2);
    t.cols = BN / 2;
  } else {
    t.n_base = g * BN;
    t.cols = BN;
  }
  return t;
}

// One CTA pair per cluster, dealt units cl, cl + clusters, ... of the
// schedule (pair_unit). A unit of `cols` columns loads cols / 2 W rows per
// CTA: map_b (128 rows), map_b_half (64), map_b_v (vn / 2) or map_b_r
// (rem / 2).
// Warps: 0 the TMA producer, 1 the MMA issuer (tensor memory owner), 2 .. 1 +
// EW the epilogue.
template <bool GATE, int EW>
__global__ void __launch_bounds__(pair_threads<EW>(), 1)
kv_proj_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_b_half,
                    const __grid_constant__ CUtensorMap map_b_v,
                    const __grid_constant__ CUtensorMap map_b_r, ple_bf16_t* __restrict__ out,
                    int M, int N, int K, const PairSched sc, int32_t* dev_err,
                    const __grid_constant__ GateEpi ge) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* a_smem = smem;
  uint8_t* b_smem = smem + P_STAGES * P_A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (P_STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * P_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + P_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t leader = rank & ~1u;       // even CTA of the pair: issues the MMAs
  const int cl = blockIdx.x / 2;
  const int num_cl = gridDim.x / 2;
  const int n_tiles = (N + BN - 1) / BN;
  const int n_groups = n_tiles;
  const int m_tiles = (M + 2 * BM - 1) / (2 * BM);
  const int num_units = sc.num_units;
  constexpr bool kStrips = EW == 8;
  const int num_kb = (K + BK * P_ATOMS - 1) / (BK * P_ATOMS);
  constexpr uint16_t pair_mask = 3u;  // both CTAs of the pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full_bar(s), 1);      // the leader's expect_tx; bytes from both CTAs
      mbar_init(empty_bar(s), 1);     // one commit of the pair leader per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * EW);  // every epilogue warp of the pair
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    // collective over the pair: the same columns in both SMs' tensor memory
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // emb (A) comes from the previous kernel
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b_half))
                 : "memory");
    if (kStrips && sc.vn > 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b_v))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b_r))
                   : "memory");
    }
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;
    bool ok = true;
    const int q = static_cast<int>(rank & 1u);  // half of the pair's rows / W tile
    for (int u = cl; ok && u < num_units; u += num_cl) {
      const PairUnit t = pair_unit<kStrips>(u, sc, n_groups, m_tiles);
      const CUtensorMap* wmap = t.cols == BN                   ? &map_b
                                : kStrips && t.cols == sc.vn ? &map_b_v
                                : t.cols == BN / 2           ? &map_b_half
                                                             : &map_b_r;
      const int m0 = t.m_base + q * BM;
      const int n0 = t.n_base + q * (t.cols / 2);
      // both CTAs' A rows and W rows of one stage
      const uint32_t stage_tx =
          kStrips ? 2u * (P_A_STAGE + static_cast<uint32_t>(P_B_STAGE / BN) *
                                          static_cast<uint32_t>(t.cols))
                  : 2u * (P_A_STAGE + (t.cols != BN ? P_B_STAGE / 2 : P_B_STAGE));
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t leader_full = map_to_rank(full_bar(stage), leader);
        if (rank == leader) {
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        }
        for (int at = 0; at < P_ATOMS; ++at) {
          const int kx = (kb * P_ATOMS + at) * BK;
          tma_load_2d_pair(smem_u32(a_smem + stage * P_A_STAGE + at * P_A_ATOM), &map_a,
                           leader_full, kx, m0);
          tma_load_2d_pair(smem_u32(b_smem + stage * P_B_STAGE + at * P_B_ATOM), wmap,
                           leader_full, kx, n0);
        }
        if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
    // The leader does not leave with copies of an armed stage in flight.
    for (int s = 0; s < P_STAGES; ++s)
      if (armed & (1u << s)) mbar_wait(full_bar(s), (armed_parity >> s) & 1u, nullptr);
  } else if (warp == 1) {
    if (rank == leader && lane == 0) {
      // ---------------- MMA issuer (pair leaders only) ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cl; ok && u < num_units; u += num_cl) {
        const uint32_t idesc = idesc_pair(pair_unit<kStrips>(u, sc, n_groups, m_tiles).cols);
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int at = 0; at < P_ATOMS; ++at) {
            const uint64_t a_desc = sw128_desc(smem_u32(a_smem + stage * P_A_STAGE + at * P_A_ATOM));
            const uint64_t b_desc = sw128_desc(smem_u32(b_smem + stage * P_B_STAGE + at * P_B_ATOM));
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint64_t koff = static_cast<uint64_t>((kk * UMMA_K * 2) >> 4);
              umma_bf16_pair(d_tmem, a_desc + koff, b_desc + koff, idesc,
                             (kb | at | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair(empty_bar(stage), pair_mask);  // frees the stage in both CTAs
          if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(accf_bar(acc), pair_mask);  // accumulator halves ready in both SMs
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
      umma_commit_pair_local(done_bar);
      mbar_wait(done_bar, 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs): this SM's 128 rows ----------------
    // Warp w reads TMEM lanes 32 (w % 4) .. +31 (its quadrant). With 8
    // warps, w and w + 4 split a tile's columns in halves, h = (w - 2) / 4;
    // of a half tile's key block (128 channels) warp h = 0 alone sums it, so
    // that every 128-channel block is one warp's, as in full tiles.
    const int quad = warp & 3;
    const int hsel = EW == 8 ? (warp - 2) >> 2 : 0;
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cl; u < num_units; u += num_cl) {
      const PairUnit t = pair_unit<kStrips>(u, sc, n_groups, m_tiles);
      const int m = t.m_base + static_cast<int>(rank & 1u) * BM + row_in_tile;
      // 8 warps: a key block's h and gammas are loaded before its MMAs end
      const bool key_block8 =
          GATE && EW == 8 && t.n_base < ge.C && (t.cols == BN || hsel == 0);
      GateBlockIn gin;
      if (key_block8) gate_block_load(ge, m, M, t.n_base + hsel * kGateBlock, lane, gin);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(accf_bar(acc), acc_phase, abort_flag));
      if (!ok) {
        if (lane == 0) { *abort_flag = 1; set_dev_err(dev_err, PLE_DEVERR_TIMEOUT); }
        break;
      }
      tc_fence_after();
      const uint32_t tlane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * ACC_COLS);
      // this warp's columns of the tile: [col0, col0 + wcols)
      const int wcols = EW == 8 ? t.cols / 2 : t.cols;
      const int col0 = hsel * wcols;
      if constexpr (GATE) {
        if (t.n_base < ge.C) {
          if (key_block8) {
            const int kc0 = hsel * kGateBlock;
            gate_block(ge, tlane + static_cast<uint32_t>(kc0), m, M, t.n_base + kc0, lane, leader,
                       acce_bar(acc), gin);
          } else if (EW == 4) {
            gate_tile(ge, tlane, m, M, t.n_base, t.cols, lane, leader, acce_bar(acc));
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar(acc), leader));
          }
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
          continue;
        }
      }
      ple_bf16_t* row_out = out + static_cast<int64_t>(m) * N;
#pragma unroll 1
      for (int chunk = 0; chunk < wcols / 32; ++chunk) {
        uint32_t r[32];
        tmem_ld32(tlane + static_cast<uint32_t>(col0 + chunk * 32), r);
        const int n = t.n_base + col0 + chunk * 32;
        if (m < M && n < N) {
          uint4* dst = reinterpret_cast<uint4*>(row_out + n);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(r[8 * q + 0], r[8 * q + 1]);
            v.y = pack_bf16x2(r[8 * q + 2], r[8 * q + 3]);
            v.z = pack_bf16x2(r[8 * q + 4], r[8 * q + 5]);
            v.w = pack_bf16x2(r[8 * q + 6], r[8 * q + 7]);
            dst[q] = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar(acc), leader));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  // No CTA leaves while its peer may still read its shared memory (the pair
  // MMAs), copy into it or arrive on its barriers.
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// 2-D K-major bf16 matrix [rows][cols], boxes of box_rows x 64 with 128-byte swizzle.
ple_status make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return fail(PLE_ERR_CUDA, "ple_kv_proj: cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                      strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PLE_ERR_CUDA, "ple_kv_proj: cuTensorMapEncodeTiled failed (%d)",
                                     static_cast<int>(r));
  return PLE_OK;
}

}  // namespace
}  // namespace ple

namespace ple {
namespace {

ple_status check_kv_args(const ple_bf16_t* emb, const ple_bf16_t* w, int64_t num_tokens,
                         int32_t emb_dim, int32_t hidden, ple_bf16_t* kv, const char* name) {
  if (num_tokens < 0 || emb_dim < 1 || hidden < 1)
    return fail(PLE_ERR_INVALID_ARG, "%s: bad sizes", name);
  if (emb_dim % 8 != 0 || hidden % 16 != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: emb_dim %% 8 and hidden %% 16 must be 0", name);
  if (num_tokens > 0x7fffffffLL - BM || 2LL * hidden > 0x7fffffffLL)
    return fail(PLE_ERR_UNSUPPORTED, "%s: sizes exceed 32-bit tile indexing", name);
  if (num_tokens == 0) return PLE_OK;
  if (!emb || !w || !kv) return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(emb) || !aligned16(w) || !aligned16(kv))
    return fail(PLE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", name);
  return PLE_OK;
}

// Launch the projection; ge != nullptr selects the fused gate epilogue
// (CTA-pair kernels only).
ple_status launch_kv(const ple_bf16_t* emb, const ple_bf16_t* w, int M, int K, int N,
                     ple_bf16_t* kv, int32_t* dev_err, cudaStream_t stream, const GateEpi* ge,
                     const char* name) {
  // Kernel: the CTA-pair kernel when there are at least two 128-row blocks
  // (always, with the fused gate), else one CTA per tile.
  // PLE_KVPROJ_MODE = pair | single overrides that choice for the plain
  // projection (launch-shape sweeps and tests); the fused gate is always
  // the pair kernel.
  bool paired = M > BM || ge != nullptr;
  if (const char* e = getenv("PLE_KVPROJ_MODE")) {
    if (strcmp(e, "single") == 0) paired = false;
    else if (strcmp(e, "pair") == 0) paired = true;
  }
  if (ge != nullptr) paired = true;
  const int cluster = paired ? 2 : 1;
  CUtensorMap map_a, map_b, map_b_half, map_b_v, map_b_r;
  ple_status s = make_map(&map_a, emb, M, K, BM);  // A rows a CTA loads
  if (s != PLE_OK) return s;
  s = make_map(&map_b, w, N, K, paired ? BN / 2 : BN);  // W rows one CTA loads per stage
  if (s != PLE_OK) return s;
  if (paired) {
    s = make_map(&map_b_half, w, N, K, BN / 4);  // a half tile's W rows per CTA
    if (s != PLE_OK) return s;
  } else {
    map_b_half = map_b;  // not read
  }
  using PairFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                          ple_bf16_t*, int, int, int, PairSched, int32_t*, GateEpi);
  // the 4-warp instantiation sizes the grid (the occupancy of both is one CTA per SM)
  using TileFn = void (*)(CUtensorMap, CUtensorMap, ple_bf16_t*, int, int, int, int32_t*);
  PairFn pair_fn = ge != nullptr ? kv_proj_pair_kernel<true, 4> : kv_proj_pair_kernel<false, 4>;
  const TileFn tile_fn = kv_proj_kernel;
  const void* fn = paired ? reinterpret_cast<const void*>(pair_fn) : reinterpret_cast<const void*>(tile_fn);
  const size_t smem = paired ? kPairSmemBytes : kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return check_cuda(err, "kv projection: smem attribute");
  // work units: 256 rows x 256 columns for the pair kernel, else 128 x 256 tiles
  int units = paired ? ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN)
                     : ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  // persistent grid: as many clusters as can be resident at once (a GPC may
  // not hold a whole number of clusters), no more than there are units
  int max_clusters = num_sms() / cluster;
  if (cluster > 1) {
    cudaLaunchConfig_t qcfg{};
    qcfg.gridDim = dim3(static_cast<unsigned>(max_clusters * cluster));
    qcfg.blockDim = dim3(paired ? pair_threads<4>() : kThreads);
    qcfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute qattr[1];
    qattr[0].id = cudaLaunchAttributeClusterDimension;
    qattr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    qattr[0].val.clusterDim.y = 1;
    qattr[0].val.clusterDim.z = 1;
    qcfg.attrs = qattr;
    qcfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, fn, &qcfg) == cudaSuccess && active > 0 &&
        active < max_clusters)
      max_clusters = active;
    cudaGetLastError();  // a failed query only leaves the SM-count bound
  }
  // Last-round split (CTA pairs): when the tiles of the last round would
  // keep at most half of the clusters busy, each of them becomes two
  // 128-column halves, so the round ends in about half the time.
  // PLE_KVPROJ_SPLIT=0 turns it off (launch-shape sweeps and tests).
  int full_units = units;
  if (paired) {
    const int rem = units % max_clusters;
    bool split = rem > 0 && 2 * rem <= max_clusters;
    if (const char* e = getenv("PLE_KVPROJ_SPLIT"))
      if (atoi(e) == 0) split = false;
    if (split) {
      full_units = units - rem;
      units = full_units + 2 * rem;
    }
  }
  const int clusters = units < max_clusters ? units : max_clusters;
  const dim3 grid(static_cast<unsigned>(clusters * cluster));
  // Few tiles per CTA pair: the 8-warp epilogue. With the fused gate, key
  // tiles first while A (emb) fits in half of L2, so that the second pass
  // over its rows (for the value tiles) reads L2, not HBM: 1024, 4096 and
  // 8192 x 2048 -> 8192 take 25.9, 77.7 and 160.1 us against 29.1, 79.9 and
  // 162.9 in the natural order on a GB300; at 32768 rows (128 MB of A) the
  // natural order is 2 % faster. PLE_KVPROJ_EPI = 4 | 8 and
  // PLE_KVPROJ_ORDER = natural | keyfirst force either choice.
  const bool few = (units + clusters - 1) / clusters <= kFewRounds;
  int epi_warps = few ? 8 : 4;
  if (const char* e = getenv("PLE_KVPROJ_EPI")) {
    if (atoi(e) == 4) epi_warps = 4;
    else if (atoi(e) == 8) epi_warps = 8;
  }
  bool key_first = ge != nullptr && static_cast<size_t>(M) * K * 2 <= kKeyFirstMaxA;
  if (const char* e = getenv("PLE_KVPROJ_ORDER")) {
    if (strcmp(e, "natural") == 0) key_first = false;
    else if (strcmp(e, "keyfirst") == 0) key_first = ge != nullptr;
  }
  const int key_groups = key_first ? ge->C / BN : 0;
  PairSched sc{full_units, key_groups, 0, 0, units};
  map_b_v = map_b_r = map_b;  // not read by the default schedule
  if (paired && key_groups > 0 && few && epi_warps == 8) {
    // Strip schedule: value strips of vn columns when, with units dealt to
    // the pairs in turn, the busiest pair then gets fewer columns (plus a
    // per-unit cost) than with the default schedule. PLE_KVPROJ_VN = 0
    // keeps the default; 128 or 192 forces that strip width.
    const int m_tiles = (M + 2 * BM - 1) / (2 * BM);
    const int C = ge->C;
    constexpr int64_t kUnitCost = 32;  // columns' worth of a unit's fixed cost
    auto busiest = [&](int n_units, auto cols_of) {
      const int P = n_units < max_clusters ? n_units : max_clusters;
      int64_t load[512] = {};
      if (P > 512) return int64_t(1) << 62;
      for (int u = 0; u < n_units; ++u) load[u % P] += cols_of(u) + kUnitCost;
      int64_t mx = 0;
      for (int p = 0; p < P; ++p) mx = load[p] > mx ? load[p] : mx;
      return mx;
    };
    auto strip_units = [&](int vn) {
      const int rem = C % vn;
      return (rem > 0 ? m_tiles : 0) + m_tiles * key_groups + m_tiles * ((C - rem) / vn);
    };
    auto strip_cols = [&](int vn) {
      const int rem = C % vn;
      const int n_rem = rem > 0 ? m_tiles : 0;
      const int n_key = m_tiles * key_groups;
      return [=](int u) { return u < n_rem ? rem : u < n_rem + n_key ? BN : vn; };
    };
    int64_t best = busiest(units, [&](int u) { return u < full_units ? BN : BN / 2; });
    int vn = 0;
    int forced = -1;
    if (const char* e = getenv("PLE_KVPROJ_VN")) forced = atoi(e);
    for (int cand : {192, 128}) {
      if (forced >= 0 && forced != cand) continue;
      const int64_t b = busiest(strip_units(cand), strip_cols(cand));
      if (forced == cand || b < best) {
        best = b;
        vn = cand;
      }
    }
    if (vn > 0) {
      sc.vn = vn;
      sc.rem = C % vn;
      sc.num_units = strip_units(vn);
      s = make_map(&map_b_v, w, N, K, vn / 2);  // a strip's W rows per CTA
      if (s != PLE_OK) return s;
      if (sc.rem > 0) {
        s = make_map(&map_b_r, w, N, K, sc.rem / 2);
        if (s != PLE_OK) return s;
      }
    }
  }
  const int launch_clusters = sc.num_units < max_clusters ? sc.num_units : max_clusters;
  const dim3 launch_grid(static_cast<unsigned>(launch_clusters * cluster));
  if (paired && epi_warps == 8) {
    pair_fn = ge != nullptr ? kv_proj_pair_kernel<true, 8> : kv_proj_pair_kernel<false, 8>;
    err = cudaFuncSetAttribute(pair_fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return check_cuda(err, "kv projection: smem attribute");
  }
  if (paired)
    err = launch_kernel(pair_fn, launch_grid,
                        dim3(epi_warps == 8 ? pair_threads<8>() : pair_threads<4>()), smem, stream,
                        static_cast<unsigned>(cluster), map_a, map_b, map_b_half, map_b_v, map_b_r,
                        kv, M, N, K, sc, dev_err, ge != nullptr ? *ge : GateEpi{});
  else
    err = launch_kernel(tile_fn, grid, dim3(kThreads), smem, stream, static_cast<unsigned>(cluster),
                        map_a, map_b, kv, M, N, K, dev_err);
  if (err != cudaSuccess) return check_cuda(err, name);
  return check_cuda(cudaGetLastError(), name);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace of ple_kv_proj_gate, B bytes: the partial sums from the start
// (16 bytes per token and 128-channel key block), the arrival counters at the end,
// counter j at 4(j+1) bytes below the end. The counters' region is sized by B
// alone -- room for one counter per 32 of the most tokens any hidden size
// could fit in B (16 bytes each) -- so every call on the same buffer and
// byte count finds its counters at the same addresses whatever its token
// count or hidden size, and no call's partial sums overlap them.
size_t gate_counter_bytes(size_t B) { return ((B / 16 + 31) / 32) * 4; }
size_t gate_partial_bytes(int64_t M, int32_t C) {
  return static_cast<size_t>(C / kGateBlock) * static_cast<size_t>(M) * 16;
}
size_t gate_ws_bytes(int64_t M, int32_t C) {
  // the smallest multiple of 256 with room for both parts (a fixed point:
  // the counters' share grows with B by 1/128 of it)
  const size_t part = gate_partial_bytes(M, C);
  size_t B = align256(part);
  for (;;) {
    const size_t need = align256(part + gate_counter_bytes(B));
    if (need <= B) return B;
    B = need;
  }
}

}  // namespace
}  // namespace ple

PLE_EXPORT ple_status ple_kv_proj(const ple_bf16_t* emb, const ple_bf16_t* w, int64_t num_tokens,
                                  int32_t emb_dim, int32_t hidden, ple_bf16_t* kv,
                                  int32_t* dev_err, cudaStream_t stream) {
  using namespace ple;
  ple_status s = check_kv_args(emb, w, num_tokens, emb_dim, hidden, kv, "ple_kv_proj");
  if (s != PLE_OK || num_tokens == 0) return s;
  return launch_kv(emb, w, static_cast<int>(num_tokens), emb_dim, 2 * hidden, kv, dev_err, stream,
                   nullptr, "ple_kv_proj launch");
}

PLE_EXPORT size_t ple_kv_proj_gate_workspace(int64_t num_tokens, int32_t hidden) {
  using namespace ple;
  if (num_tokens <= 0 || hidden < BN || hidden % BN != 0) return 0;
  return gate_ws_bytes(num_tokens, hidden);
}

PLE_EXPORT ple_status ple_kv_proj_gate(const ple_bf16_t* emb, const ple_bf16_t* w,
                                       int64_t num_tokens, int32_t emb_dim, int32_t hidden,
                                       const ple_bf16_t* hidden_states, const ple_bf16_t* gamma_h,
                                       const ple_bf16_t* gamma_k, float eps, ple_bf16_t* kv,
                                       float* gate_out, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_err, cudaStream_t stream) {
  using namespace ple;
  const char* name = "ple_kv_proj_gate";
  ple_status s = check_kv_args(emb, w, num_tokens, emb_dim, hidden, kv, name);
  if (s != PLE_OK) return s;
  if (hidden % BN != 0)
    return fail(PLE_ERR_UNSUPPORTED, "%s: hidden_size %d must be a multiple of %d", name, hidden, BN);
  if (num_tokens == 0) return PLE_OK;
  if (!hidden_states || !gamma_h || !gamma_k || !gate_out || !workspace)
    return fail(PLE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(hidden_states) || !aligned16(gamma_h) || !aligned16(gamma_k) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PLE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned (workspace 256)", name);
  if (gate_partial_bytes(num_tokens, hidden) + gate_counter_bytes(workspace_bytes) >
      workspace_bytes)
    return fail(PLE_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name,
                workspace_bytes, gate_ws_bytes(num_tokens, hidden));
  GateEpi ge{};
  ge.hidden = hidden_states;
  ge.gamma_h = gamma_h;
  ge.gamma_k = gamma_k;
  ge.partial = static_cast<float4*>(workspace);
  ge.count_top = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) +
                                             (workspace_bytes & ~static_cast<size_t>(3)));
  ge.gate_out = gate_out;
  ge.eps = eps;
  ge.C = hidden;
  return launch_kv(emb, w, static_cast<int>(num_tokens), emb_dim, 2 * hidden, kv, dev_err, stream,
                   &ge, "ple_kv_proj_gate launch");
}
