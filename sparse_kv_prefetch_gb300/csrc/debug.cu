// Test hooks.  Neither is part of the decode step; both exist so that tests
// can perturb and probe it without faulting or hanging the GPU.
//
// delay_kernel: one thread sleeps (__nanosleep) until `ns` nanoseconds of the
//   global timer have passed; launched on one stream it holds back the work
//   queued after it there, so tests can check that a schedule's events, not
//   luck, order its kernels.  Bounded by ns (at most 100 ms).
// expire_kernel: one thread waits on a shared-memory mbarrier that nothing
//   ever arrives at, with the same bounded wait every kernel of the library
//   uses, here with a short limit; when it gives up it sets the status word
//   that dd_check_device reports as DD_ERR_TIMEOUT, then returns normally.
#include "dd_internal.cuh"

namespace dd {
namespace {

__device__ unsigned int g_debug_status = 0;

__global__ void delay_kernel(uint64_t ns) {
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < ns) __nanosleep(1000);
}

__global__ void expire_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  mbar_fence_init();
  if (!mbar_wait_for(&bar, 0, limit_ns)) atomicOr(&g_debug_status, 1u);
}

}  // namespace

constexpr uint64_t kMaxDebugNs = 100000000ull;  // 100 ms

cudaError_t launch_delay(uint64_t ns, cudaStream_t st) {
  delay_kernel<<<1, 1, 0, st>>>(ns < kMaxDebugNs ? ns : kMaxDebugNs);
  return cudaGetLastError();
}

cudaError_t launch_expire_wait(uint64_t limit_ns, cudaStream_t st) {
  expire_kernel<<<1, 1, 0, st>>>(limit_ns < kMaxDebugNs ? limit_ns : kMaxDebugNs);
  return cudaGetLastError();
}

unsigned int take_debug_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_debug_status, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_debug_status, &zero, sizeof zero);
  return v;
}

}  // namespace dd
