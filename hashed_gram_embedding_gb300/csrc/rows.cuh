// Row-vector helpers of the gather kernels (ple_lookup and its variants in
// lookup.cu, the sharded gather and the row selection in shard.cu): one
// 16-byte table vector per load, and the fp8 e4m3 dequantisation of 16 codes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace ple {

// One 16-byte vector of a table row: read-only path, no L1 allocation, the
// whole 256-byte L2 sector group requested (the rest of the row follows).
__device__ __forceinline__ uint4 load_row_vec(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Two e4m3 codes -> two bf16 values, bf16_rn(float(e4m3) * scale): the
// codes widen exactly (through half), one float32 product each, then
// round-to-nearest-even to bf16.
__device__ __forceinline__ uint32_t dequant_pair(uint16_t codes, float scale) {
  const __half2 h2(__nv_cvt_fp8x2_to_halfraw2(codes, __NV_E4M3));
  const float2 f = __half22float2(h2);
  const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 16 codes (one vector) -> 16 bf16 values (two vectors, lo = codes 0..7).
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

}  // namespace ple
