// Tensor-memory-access (TMA) helpers shared by the kernels that stage tiles
// with cp.async.bulk.tensor: the driver's tensor-map encoder (resolved at
// run time, so the library links no libcuda) and the tiled 2-D load.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ple {

// cuTensorMapEncodeTiled of the installed driver, or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// TMA copy of the box at (x, y) of a 2-D tensor map into this CTA's shared
// memory, its bytes counted on the mbarrier at shared address bar. x is an
// element index whose byte offset must be a multiple of 16; boxes may start
// at negative or out-of-range coordinates (those elements read as zero).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Expect `bytes` more transaction bytes on an mbarrier's current phase
// without arriving on it.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

}  // namespace ple
