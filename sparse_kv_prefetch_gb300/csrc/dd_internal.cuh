// Internal declarations shared by the kernels and the C-ABI layer of libdd.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dd.h"

namespace dd {

// Resolved shape of one layer plus the derived launch geometry.
struct Dims {
  int B, Hq, Hkv, G, d, n, k, W, dtype;
  int U;        // units = B * Hkv
  int span;     // candidate positions [0, n - W)
  int ldn;      // row stride of the fp32 logits (n rounded up to 4)
  int chunk;    // keys per scoring CTA
  int nchunks;  // scoring CTAs per unit
  int rows;     // attended rows per unit = k + W
  int nsplit;   // split-k attention CTAs per unit
  int elt;      // bytes per stored element
};

// Byte offsets of the workspace regions (each 256-byte aligned).
struct WsLayout {
  size_t logits, part, attn_o, attn_ml, total;
};

dd_status resolve(const dd_shape* s, Dims* out);
WsLayout ws_layout(const Dims& d);

constexpr int kAttnRowsPerSplit = 64;

// Kernel launchers (score.cu, topk.cu, gather.cu, attn.cu).  Each returns the
// launch status (cudaGetLastError after the launch).
cudaError_t launch_score(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, cudaStream_t st);
cudaError_t launch_topk(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                        float* sel, float* lse, cudaStream_t st);
cudaError_t launch_gather(const Dims& d, const void* k_host, const void* v_host,
                          const int32_t* idx, void* k_buf, void* v_buf, cudaStream_t st);
cudaError_t launch_attn(const Dims& d, const void* q, const void* k_buf, const void* v_buf,
                        const void* k_dev, const void* v_win, float* out, float* part_o,
                        float2* part_ml, cudaStream_t st);

// Number of kernels each launcher enqueues.
constexpr int kScoreLaunches = 1, kTopkLaunches = 1, kGatherLaunches = 1, kAttnLaunches = 2;

int sm_count();

// Keys per scoring CTA for a stored dtype and head size (0 if unsupported).
int score_chunk(int dtype, int head_dim);

// ----------------------------------------------------------------- device

// Rows of K / V are moved as 16-byte vectors: 8 bf16 or 4 fp32 elements.
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
};
struct bf16_t {
  uint16_t bits;
};
template <>
struct Elem<bf16_t> {
  static constexpr int kVec = 8;
};

// Widen one 16-byte vector into fp32 values (bf16 -> fp32 is exact: the
// bf16 bits are the upper half of the binary32 pattern).
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

// Streaming 16-byte load: read once, evict first (keeps L2 for reused data).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
// Read-only 16-byte load through the non-coherent path.
__device__ __forceinline__ uint4 ld_ro(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Merge two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(m, a.y * __expf(a.x - m) + b.y * __expf(b.x - m));
}

}  // namespace dd
