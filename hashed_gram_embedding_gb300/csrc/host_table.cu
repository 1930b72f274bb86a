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
// kernel cannot supply huge pages the memory still works, only slower. The
// mapping also gets an explicit NUMA policy (the calling CPU's node,
// preferred), which keeps automatic NUMA balancing from periodically
// unmapping its pages under the GPU's reads.
#include "common.cuh"

#include <fcntl.h>
#include <sched.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <sys/syscall.h>
#include <unistd.h>
#include <cerrno>
#include <cstring>

namespace {
constexpr size_t kAlign = size_t(1) << 30;  // covers 2 MiB and 512 MiB huge pages

// An explicit memory policy for a mapping (prefer the calling CPU's NUMA
// node): the kernel's automatic NUMA balancing only scans mappings without
// one, and its periodic unmapping of sampled pages would make the GPU's reads
// of those pages take slow translation faults. Advisory.
void prefer_local_node(void* p, size_t bytes) {
  unsigned cpu = 0, node = 0;
  if (syscall(SYS_getcpu, &cpu, &node, nullptr) == 0 && node < 64) {
    const unsigned long mask = 1ul << node;
    constexpr int kMpolPreferred = 1;
    syscall(SYS_mbind, p, bytes, kMpolPreferred, &mask, 64ul, 0u);
  }
}

// A POSIX shared-memory name: "/" then 1..254 characters, no other "/".
bool valid_shm_name(const char* name) {
  if (name == nullptr || name[0] != '/') return false;
  const size_t n = strlen(name);
  if (n < 2 || n > 255) return false;
  return strchr(name + 1, '/') == nullptr;
}

// Register [p, p+bytes) for GPU access when asked; on failure the mapping is
// left to the caller to undo.
ple_status maybe_register(void* p, size_t bytes, int32_t flags, unsigned extra,
                          const char* what) {
  if ((flags & PLE_HOST_TABLE_REGISTER) == 0) return PLE_OK;
  cudaError_t err = cudaHostRegister(p, bytes, cudaHostRegisterPortable |
                                                   cudaHostRegisterMapped | extra);
  return ple::check_cuda(err, what);
}

// Map a shared-memory object (created or existing) and register it.
ple_status map_shared(const char* name, size_t bytes, int32_t flags, bool create,
                      void** host_ptr, const char* fn) {
  using namespace ple;
  if (host_ptr == nullptr) return fail(PLE_ERR_INVALID_ARG, "%s: null out pointer", fn);
  *host_ptr = nullptr;
  if (!valid_shm_name(name))
    return fail(PLE_ERR_INVALID_ARG, "%s: name must be \"/\" then 1..254 characters, no \"/\"", fn);
  if (bytes == 0) return fail(PLE_ERR_INVALID_ARG, "%s: zero bytes", fn);
  const int fd = shm_open(name, create ? (O_RDWR | O_CREAT | O_EXCL) : O_RDWR, 0600);
  if (fd < 0) return fail(PLE_ERR_INVALID_ARG, "%s: shm_open(%s): %s", fn, name, strerror(errno));
  auto undo = [&](void* m) {  // roll back everything this call did
    if (m != nullptr && m != MAP_FAILED) munmap(m, bytes);
    close(fd);
    if (create) shm_unlink(name);
  };
  if (create) {
    if (ftruncate(fd, static_cast<off_t>(bytes)) != 0) {
      const int e = errno;
      undo(nullptr);
      return fail(PLE_ERR_CUDA, "%s: sizing %s to %zu bytes: %s", fn, name, bytes, strerror(e));
    }
  } else {
    struct stat st {};
    if (fstat(fd, &st) != 0 || static_cast<size_t>(st.st_size) < bytes) {
      undo(nullptr);
      return fail(PLE_ERR_INVALID_ARG, "%s: %s holds fewer than %zu bytes", fn, name, bytes);
    }
  }
  void* m = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_SHARED, fd, 0);
  if (m == MAP_FAILED) {
    const int e = errno;
    undo(m);
    return fail(PLE_ERR_CUDA, "%s: mmap of %s: %s", fn, name, strerror(e));
  }
  madvise(m, bytes, MADV_HUGEPAGE);  // shared-memory huge pages, where enabled
  prefer_local_node(m, bytes);
  ple_status s = maybe_register(m, bytes, flags, 0u, fn);
  if (s != PLE_OK) {
    undo(m);
    return s;
  }
  close(fd);  // the mapping keeps the object alive
  *host_ptr = m;
  return PLE_OK;
}
}  // namespace

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
  prefer_local_node(p, bytes);
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

PLE_EXPORT ple_status ple_host_table_create_shared(const char* name, size_t bytes, int32_t flags,
                                                   void** host_ptr) {
  return map_shared(name, bytes, flags, true, host_ptr, "ple_host_table_create_shared");
}

PLE_EXPORT ple_status ple_host_table_attach_shared(const char* name, size_t bytes, int32_t flags,
                                                   void** host_ptr) {
  return map_shared(name, bytes, flags, false, host_ptr, "ple_host_table_attach_shared");
}

PLE_EXPORT ple_status ple_host_table_unlink_shared(const char* name) {
  using namespace ple;
  if (!valid_shm_name(name))
    return fail(PLE_ERR_INVALID_ARG, "ple_host_table_unlink_shared: bad name");
  if (shm_unlink(name) != 0)
    return fail(PLE_ERR_INVALID_ARG, "ple_host_table_unlink_shared(%s): %s", name, strerror(errno));
  return PLE_OK;
}

PLE_EXPORT ple_status ple_host_table_map_file(const char* path, size_t bytes, int32_t flags,
                                              void** host_ptr) {
  using namespace ple;
  const char* fn = "ple_host_table_map_file";
  if (host_ptr == nullptr) return fail(PLE_ERR_INVALID_ARG, "%s: null out pointer", fn);
  *host_ptr = nullptr;
  if (path == nullptr || bytes == 0) return fail(PLE_ERR_INVALID_ARG, "%s: bad arguments", fn);
  const int fd = open(path, O_RDONLY);
  if (fd < 0) return fail(PLE_ERR_INVALID_ARG, "%s: open(%s): %s", fn, path, strerror(errno));
  struct stat st {};
  if (fstat(fd, &st) != 0 || static_cast<size_t>(st.st_size) < bytes) {
    close(fd);
    return fail(PLE_ERR_INVALID_ARG, "%s: %s holds fewer than %zu bytes", fn, path, bytes);
  }
  void* m = mmap(nullptr, bytes, PROT_READ, MAP_SHARED, fd, 0);
  if (m == MAP_FAILED) {
    const int e = errno;
    close(fd);
    return fail(PLE_ERR_CUDA, "%s: mmap of %s: %s", fn, path, strerror(e));
  }
  madvise(m, bytes, MADV_RANDOM);  // rows are read in no particular order
  cudaError_t rerr = cudaSuccess;
  if (flags & PLE_HOST_TABLE_REGISTER) {
    rerr = cudaHostRegister(m, bytes, cudaHostRegisterPortable | cudaHostRegisterMapped |
                                          cudaHostRegisterReadOnly);
    if (rerr == cudaErrorNotSupported) {
      // Read-only registration is not available on every platform: map the
      // file privately instead (pinning gives each page its own copy, so the
      // file is read once into memory) and register that.
      cudaGetLastError();
      munmap(m, bytes);
      m = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE, fd, 0);
      if (m == MAP_FAILED) {
        const int e = errno;
        close(fd);
        return fail(PLE_ERR_CUDA, "%s: private mmap of %s: %s", fn, path, strerror(e));
      }
      madvise(m, bytes, MADV_RANDOM);
      rerr = cudaHostRegister(m, bytes, cudaHostRegisterPortable | cudaHostRegisterMapped);
    }
  }
  close(fd);  // the mapping keeps the file open
  if (rerr != cudaSuccess) {
    munmap(m, bytes);
    return check_cuda(rerr, fn);
  }
  *host_ptr = m;
  return PLE_OK;
}

PLE_EXPORT ple_status ple_host_table_unmap(void* host_ptr, size_t bytes, int32_t flags) {
  using namespace ple;
  if (host_ptr == nullptr) return PLE_OK;
  cudaError_t err = cudaSuccess;
  if (flags & PLE_HOST_TABLE_REGISTER) err = cudaHostUnregister(host_ptr);
  munmap(host_ptr, bytes);
  return check_cuda(err, "ple_host_table_unmap: cudaHostUnregister");
}
