// Host KV store allocators of libdd.so and the translation of host-store
// pointers for the gather.
//
// The gather reads the selected rows straight out of host memory (DualDecoder
// paper, Sec. 2.2: the KV cache lives in host memory and only the selected
// entries cross the host-to-device link).  How the GPU translates those host
// addresses decides how fast a scattered gather can go, and how much it slows
// the kernels running beside it: every distinct page a gather touches needs a
// translation, and with the host's 64 KiB base pages a long-context layer
// touches hundreds of thousands of them.  dd_host_alloc gives the store
// transparent huge pages instead: anonymous memory, faulted in from the CPU,
// locked (mlock) and registered with CUDA (cudaHostRegister).
// dd_host_alloc_pinned is the alternative that stays put: page-locked memory
// the CUDA driver allocates itself (cudaHostAlloc), in the host's base pages.
// On the GB300 hosts measured, huge-page stores had pages split and moved by
// the host now and then, whatever the locking, and every read of the store
// from the GPU slowed to a few GB/s while that lasted; driver-allocated
// memory never did.
//
// Any page-locked host memory known to CUDA (torch pin_memory,
// cudaHostAlloc) works with the gather as well.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <sys/mman.h>

#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <thread>
#include <vector>

#ifndef DD_HOST_PREFAULT
#define DD_HOST_PREFAULT 1
#endif

#include "dd_internal.cuh"

namespace dd {

size_t host_page_bytes() {
  static size_t cached = 0;
  if (cached) return cached;
  size_t v = 0;
  if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long x = 0;
    if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
    std::fclose(f);
  }
  if (v < 4096 || (v & (v - 1))) v = (size_t)2 << 20;
  cached = v;
  return v;
}

namespace {

enum Kind { kHuge = 1, kPinned = 2 };

struct Region {
  size_t len;   // bytes the caller may use
  int kind;
  bool locked;  // kHuge: mlock succeeded
};

std::mutex g_mu;
std::map<uintptr_t, Region> g_regions;  // base address -> region

// The region holding p, if any (under g_mu).
const Region* find_region(const void* p, uintptr_t* base) {
  auto it = g_regions.upper_bound((uintptr_t)p);
  if (it == g_regions.begin()) return nullptr;
  --it;
  if ((uintptr_t)p >= it->first + it->second.len) return nullptr;
  if (base) *base = it->first;
  return &it->second;
}

}  // namespace

bool in_huge_page_store(const void* p) {
  std::lock_guard<std::mutex> lock(g_mu);
  const Region* r = find_region(p, nullptr);
  return r && r->kind == kHuge;
}

const void* host_to_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the non-sticky error
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost) return nullptr;
  return a.devicePointer;
}

}  // namespace dd

using namespace dd;

extern "C" {

dd_status dd_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return DD_ERR_INVALID_ARG;
  *out = nullptr;
  const size_t page = host_page_bytes();
  const size_t len = (bytes + page - 1) / page * page;
  // Over-map by one huge page so the region can start on a huge-page boundary.
  void* raw = mmap(nullptr, len + page, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED) return DD_ERR_OOM;
  const uintptr_t r = (uintptr_t)raw;
  const uintptr_t base = (r + page - 1) / page * page;
  if (base > r) munmap(raw, base - r);
  const uintptr_t tail = base + len, raw_end = r + len + page;
  if (raw_end > tail) munmap((void*)tail, raw_end - tail);
  void* p = (void*)base;
  madvise(p, len, MADV_HUGEPAGE);  // advisory: huge pages where the host allows them
#if DD_HOST_PREFAULT
  // Fault the region in from the CPU (one store per 64 KiB, several threads,
  // each on its own huge pages) before registering it, so that the kernel
  // backs it with huge pages at first touch.
  {
    const unsigned hw = std::thread::hardware_concurrency();
    const size_t n_pages = len / page;
    const unsigned n_thr = (unsigned)std::min<size_t>(n_pages, hw ? std::min(hw, 16u) : 4u);
    auto fault = [&](unsigned t) {
      for (size_t pg = t; pg < n_pages; pg += n_thr)
        for (size_t off = 0; off < page; off += 65536)
          static_cast<volatile unsigned char*>(p)[pg * page + off] = 0;
    };
    std::vector<std::thread> th;
    for (unsigned t = 1; t < n_thr; ++t) th.emplace_back(fault, t);
    fault(0);
    for (auto& x : th) x.join();
  }
#endif
  // Lock the region before registering it.  Without the lock, once the CPU
  // has written a store (the caller filling it) the host kernel split some of
  // its huge pages and migrated pages when the GPU began reading it, and
  // every gather over the store slowed to a few GB/s for as long as that
  // went on.  Locked pages stay put.  Best effort: without the privilege to
  // lock this much memory the store is still registered and used.
  const bool locked = mlock(p, len) == 0;
  if (cudaHostRegister(p, len, cudaHostRegisterDefault) != cudaSuccess) {
    cudaGetLastError();
    if (locked) munlock(p, len);
    munmap(p, len);
    return DD_ERR_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_regions[(uintptr_t)p] = Region{len, kHuge, locked};
  }
  *out = p;
  return DD_OK;
}

dd_status dd_host_alloc_pinned(size_t bytes, void** out) {
  if (!out || bytes == 0) return DD_ERR_INVALID_ARG;
  *out = nullptr;
  void* p = nullptr;
  if (cudaHostAlloc(&p, bytes, cudaHostAllocPortable) != cudaSuccess || !p) {
    cudaGetLastError();
    return DD_ERR_OOM;
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_regions[(uintptr_t)p] = Region{bytes, kPinned, false};
  }
  *out = p;
  return DD_OK;
}

dd_status dd_host_free(void* p) {
  if (!p) return DD_OK;
  Region r;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_regions.find((uintptr_t)p);
    if (it == g_regions.end()) return DD_ERR_INVALID_ARG;
    r = it->second;
    g_regions.erase(it);
  }
  if (r.kind == kPinned) return cudaFreeHost(p) == cudaSuccess ? DD_OK : DD_ERR_CUDA;
  const cudaError_t e = cudaHostUnregister(p);
  if (r.locked) munlock(p, r.len);
  munmap(p, r.len);
  return e == cudaSuccess ? DD_OK : DD_ERR_CUDA;
}

size_t dd_host_page_bytes(void) { return host_page_bytes(); }

int dd_host_store_kind(const void* p) {
  std::lock_guard<std::mutex> lock(g_mu);
  const Region* r = find_region(p, nullptr);
  return r ? r->kind : 0;
}

int dd_host_store_locked(const void* p) {
  std::lock_guard<std::mutex> lock(g_mu);
  const Region* r = find_region(p, nullptr);
  return r && r->locked ? 1 : 0;
}

}  // extern "C"
