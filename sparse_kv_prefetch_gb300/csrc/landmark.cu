// Landmark (chunk) selection.  The DualDecoder paper computes the retrieval
// index from the token being processed and static GPU-resident KV landmarks
// (Sec. 1); Sec. 2.2 describes chunks of adjacent KV entries with compressed
// landmarks, the GPU selecting chunks for the current query and retrieving
// their entries from host memory.  Here a landmark is the mean key of a chunk
// of c adjacent positions of [0, n - W), kept in fp32 in HBM (c times smaller
// than K in elements).  Selection scores the landmarks with the scoring and
// top-k kernels (as a key cache of M = (n - W) / c rows; the scoring kernel
// widens a bf16 query itself) and the top-k writes each of the k / c selected
// chunks as its c rows, which the gather then moves as runs of c contiguous
// rows.
//
// landmark_kernel: one thread per (unit, chunk, 16-byte piece of a row); it
//   sums the piece over the chunk's c rows in fp32 and divides by c.
// For the fused form of steps 1-2 (DD_STEP_FUSED_TOPK), whose scoring kernel
// takes an fp32 query and writes chunk ids:
// to_f32_kernel: widens bf16 queries to fp32;
// expand_kernel: rows[u][i c + r] = chunk[u][i] c + r.
#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kLmThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kLmThreads)
    landmark_kernel(const uint4* __restrict__ K, float4* __restrict__ L, int n, int chunk, int M,
                    long long total) {
  constexpr int VEC = Elem<T>::kVec, LPR = D / VEC;  // 16-byte pieces per K row
  const long long t = (long long)blockIdx.x * kLmThreads + threadIdx.x;
  if (t >= total) return;
  const int part = (int)(t % LPR);
  const long long um = t / LPR;
  const long long u = um / M;
  const int m = (int)(um - u * M);
  const uint4* src = K + ((size_t)u * n + (size_t)m * chunk) * LPR + part;
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int r = 0; r < chunk; ++r) {
    float f[VEC];
    unpack(ld_ro(src + (size_t)r * LPR), f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] += f[e];
  }
  const float cf = (float)chunk;
  float4* dst = L + ((size_t)um * D + (size_t)part * VEC) / 4;
#pragma unroll
  for (int e = 0; e < VEC; e += 4)
    dst[e / 4] = make_float4(acc[e] / cf, acc[e + 1] / cf, acc[e + 2] / cf, acc[e + 3] / cf);
}

__global__ void expand_kernel(const int32_t* __restrict__ chunks, int32_t* __restrict__ rows,
                              int chunk, long long total) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const long long i = t / chunk;  // (unit, selected chunk) pair
  const int r = (int)(t - i * chunk);
  rows[t] = chunks[i] * chunk + r;
}

__global__ void to_f32_kernel(const uint16_t* __restrict__ x, float* __restrict__ y, int count) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < count) y[t] = __uint_as_float((uint32_t)x[t] << 16);
}

template <typename T, int D>
cudaError_t launch_lm(const Dims& d, int chunk, const void* k_dev, float* L, cudaStream_t st) {
  constexpr int LPR = D / Elem<T>::kVec;
  const int M = d.span / chunk;
  const long long total = (long long)d.U * M * LPR;
  const long long grid = (total + kLmThreads - 1) / kLmThreads;
  landmark_kernel<T, D><<<(unsigned)grid, kLmThreads, 0, st>>>(
      static_cast<const uint4*>(k_dev), reinterpret_cast<float4*>(L), d.n, chunk, M, total);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_landmarks(const Dims& d, int chunk, const void* k_dev, float* landmarks,
                             cudaStream_t st) {
  if (d.dtype == DD_BF16) {
    if (d.d == 64) return launch_lm<bf16_t, 64>(d, chunk, k_dev, landmarks, st);
    if (d.d == 128) return launch_lm<bf16_t, 128>(d, chunk, k_dev, landmarks, st);
  } else {
    if (d.d == 64) return launch_lm<float, 64>(d, chunk, k_dev, landmarks, st);
    if (d.d == 128) return launch_lm<float, 128>(d, chunk, k_dev, landmarks, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_expand(const int32_t* chunks, int32_t* rows, int units, int kc, int chunk,
                          cudaStream_t st) {
  const long long total = (long long)units * kc * chunk;
  const unsigned grid = (unsigned)((total + 255) / 256);
  expand_kernel<<<grid, 256, 0, st>>>(chunks, rows, chunk, total);
  return cudaGetLastError();
}

cudaError_t launch_to_f32(const void* x_bf16, float* y, int count, cudaStream_t st) {
  to_f32_kernel<<<(count + 255) / 256, 256, 0, st>>>(static_cast<const uint16_t*>(x_bf16), y,
                                                     count);
  return cudaGetLastError();
}

}  // namespace dd
