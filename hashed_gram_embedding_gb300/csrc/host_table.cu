// ple_host_table_alloc / ple_host_table_free: host memory for a PLE table
// that the GPU reads in place over UVA.
//
// Source: PR#54371 report ("Support UVA PLE-offload ..."), 关键源码片段
// (the pinned-host backend allocates the weight in pinned memory and the GPU
// reads the rows it needs directly through UVA); PR#56512 report, 关键源码片段
// (a shared table mapped into the process and registered with
// cudaHostRegister).
//
// Why not cudaHostAlloc: a row gather touches ids spread uniformly over the
// whole table. With small pages every row of a multi-GB table is a different
// GPU address translation, and translation misses, not the host link, then
// bound the gather (a few GB/s measured). The memory here is an anonymous
// mapping aligned to 1 GiB and advised for transparent huge pages
// (madvise(MADV_HUGEPAGE)) before cudaHostRegister pins it, so the GPU maps
// it with huge pages and a random gather runs near the link rate. If the
// kernel cannot supply huge pages the memory still works, only slower.
#include "common.cuh"

#include <sys/mman.h>
#include <cerrno>
#include <cstring>

namespace {
constexpr size_t kAlign = size_t(1) << 30;  // covers 2 MiB and 512 MiB huge pages
}

PLE_EXPORT ple_status ple_host_table_alloc(size_t bytes, void** host_ptr) {
  using namespace ple;
  if (host_ptr == nullptr) return fail(PLE_ERR_INVALID_ARG, "ple_host_table_alloc: null out pointer");
  *host_ptr = nullptr;
  if (bytes == 0) return fail(PLE_ERR_INVALID_ARG, "ple_host_table_alloc: zero bytes");
  const size_t span = bytes + kAlign;
  void* base = mmap(nullptr, span, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (base == MAP_FAILED)
    return fail(PLE_ERR_CUDA, "ple_host_table_alloc: mmap of %zu bytes failed: %s", span,
                strerror(errno));
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  const uintptr_t aligned = (b + kAlign - 1) & ~(static_cast<uintptr_t>(kAlign) - 1);
  // keep exactly [aligned, aligned + bytes) mapped
  if (aligned > b) munmap(base, aligned - b);
  const uintptr_t end = aligned + bytes;
  const uintptr_t map_end = b + span;
  if (map_end > end) munmap(reinterpret_cast<void*>(end), map_end - end);
  void* p = reinterpret_cast<void*>(aligned);
  madvise(p, bytes, MADV_HUGEPAGE);  // advisory: failure only costs speed
  // Fault the memory in from the CPU first, one byte per 2 MiB: with the
  // advice in place each fault maps a whole huge page (pinning alone may
  // populate small pages).
  volatile uint8_t* bytes_p = static_cast<volatile uint8_t*>(p);
  for (size_t off = 0; off < bytes; off += size_t(2) << 20) bytes_p[off] = 0;
  cudaError_t err = cudaHostRegister(p, bytes, cudaHostRegisterPortable | cudaHostRegisterMapped);
  if (err != cudaSuccess) {
    munmap(p, bytes);
    return check_cuda(err, "ple_host_table_alloc: cudaHostRegister");
  }
  *host_ptr = p;
  return PLE_OK;
}

PLE_EXPORT ple_status ple_host_table_free(void* host_ptr, size_t bytes) {
  using namespace ple;
  if (host_ptr == nullptr) return PLE_OK;
  cudaError_t err = cudaHostUnregister(host_ptr);
  munmap(host_ptr, bytes);
  return check_cuda(err, "ple_host_table_free: cudaHostUnregister");
}
