// dd_sparse_decode_attn_noalloc: the split-k attention of dd_sparse_decode_attn
// for callers that cannot allocate device memory at all, not even a caller-
// owned workspace.  Examples: an engine that has promised every free byte of
// HBM to its KV-cache pool, or a plugin inside a framework that owns all
// device allocations.  It also helps loops that must not stall the GPU:
// cudaMalloc synchronises the device.
//
// Its only scratch, the per-split partials (o, max, sum of exp), lives in a
// file-scope device array of DD_NOALLOC_SCRATCH_BYTES.  The array is part of
// the library image: every GPU that loads libdd.so holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, so its
// device address is looked up with cudaGetSymbolAddress, once per device, on
// the first call made with that device current; that first call should come
// before any stream capture.
//
// Every call shares the one array, which keeps the last call's contents.
// Nothing in it needs to start at zero: each split writes its partial before
// the merge kernel reads it.  Calls that overlap on the GPU (two streams, or
// two host threads) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dd_internal.cuh"

namespace {

using dd::Dims;

static __device__ __align__(256) unsigned char g_attn_scratch[DD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_dev[kMaxDevices] = {};  // device address of g_attn_scratch, per device

// Device address of the scratch array on the current device (looked up once).
dd_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DD_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return DD_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" dd_status dd_sparse_decode_attn_noalloc(const dd_shape* shape, const void* q,
                                                   const void* k_buf, const void* v_buf,
                                                   const void* k_dev, const void* v_win,
                                                   float* out, dd_stream_t stream) {
  Dims d;
  dd_status st = dd::resolve(shape, &d);
  if (st != DD_OK) return st;
  // Partials: o [B*H_q][nsplit][d] fp32 (256-byte aligned), then (max, sum) pairs.
  const size_t o_bytes =
      (((size_t)d.B * d.Hq * d.nsplit * d.d * sizeof(float)) + 255) & ~(size_t)255;
  const size_t ml_bytes = (size_t)d.B * d.Hq * d.nsplit * sizeof(float2);
  if (o_bytes + ml_bytes > (size_t)DD_NOALLOC_SCRATCH_BYTES) return DD_ERR_UNSUPPORTED;
  if (!q || !k_buf || !v_buf || !k_dev || !out) return DD_ERR_INVALID_ARG;
  if (d.W > 0 && !v_win) return DD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(k_dev) ||
      !aligned16(out) || (v_win && !aligned16(v_win)))
    return DD_ERR_INVALID_ARG;
  // The same pointer check as every other entry point: device memory of the
  // current device (or managed memory).
  if (!dd::all_device({q, k_buf, v_buf, k_dev, v_win, static_cast<const void*>(out)}))
    return DD_ERR_INVALID_ARG;
  void* base = nullptr;
  st = scratch_address(&base);
  if (st != DD_OK) return st;
  char* b = static_cast<char*>(base);
  const cudaError_t e =
      dd::launch_attn(d, q, k_buf, v_buf, dd::window_in_cache(k_dev, d), v_win, out, reinterpret_cast<float*>(b),
                      reinterpret_cast<float2*>(b + o_bytes), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DD_OK : DD_ERR_CUDA;
}
