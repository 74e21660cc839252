// Step 1 of the decode step: score the speculated token's query against the
// key cache, s[b,h,j] = q_spec[b,h] . K[b,h_kv,j] / sqrt(d), together with the
// online softmax statistics (max, sum of exp) of every chunk of positions.
// (DualDecoder summary page, core formulas: alpha = softmax(q_spec K^T /
// sqrt(d_k)); paper Sec. 1: the retrieval index is computed from the token
// being processed and the key cache.)
//
// The kernel is HBM-bound: every K row is read exactly once, 2 flops per
// element.  Each group of LPR lanes owns one K row per load (LPR x 16 bytes =
// d elements), a lane keeps U rows in flight, and the lane group reduces the
// partial dot products with xor-shuffles.  All query heads of a GQA group are
// scored from the same K load.
#include <math.h>

#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kRowsInFlight = 8;  // U: rows per lane group per iteration
constexpr int kItersPerChunk = 8;

template <typename T, int D>
struct ScoreGeom {
  static constexpr int kVec = Elem<T>::kVec;
  static constexpr int kLpr = D / kVec;          // lanes per row
  static constexpr int kRpw = 32 / kLpr;         // rows per warp per load
  static constexpr int kGroups = kScoreWarps * kRpw;
  static constexpr int kRowsIt = kGroups * kRowsInFlight;
  static constexpr int kChunk = kRowsIt * kItersPerChunk;
  static_assert(kLpr >= kRowsInFlight && kLpr <= 32, "unsupported row width");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kScoreThreads)
    score_kernel(const uint4* __restrict__ q_spec, const uint4* __restrict__ K,
                 float* __restrict__ logits, float2* __restrict__ part, int n, int ldn, int Hq,
                 int Hkv, int nchunks, float scale) {
  using Geo = ScoreGeom<T, D>;
  constexpr int VEC = Geo::kVec, LPR = Geo::kLpr, RPW = Geo::kRpw;
  constexpr int NG = Geo::kGroups, U = kRowsInFlight;
  constexpr int V16 = D / VEC;  // 16-byte vectors per row (== LPR)

  const int item = blockIdx.x;
  const int u = item / nchunks, c = item - u * nchunks;
  const int b = u / Hkv, hk = u - b * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPR;
  const int grp = warp * RPW + lane / LPR;

  // This lane's slice of each query head of the group, in fp32.
  float qf[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 v = ld_ro(q_spec + ((size_t)(b * Hq + hk * G + g)) * V16 + sub);
    unpack(v, qf[g]);
  }

  const uint4* Ku = K + (size_t)u * n * V16;
  const int j_begin = c * Geo::kChunk;
  const int j_end = min(n, j_begin + Geo::kChunk);

  float m_run[G], l_run[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.f;
  }

  for (int base = j_begin; base < j_end; base += Geo::kRowsIt) {
    uint4 v[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int j = base + i * NG + grp;
      v[i] = (j < j_end) ? ld_stream(Ku + (size_t)j * V16 + sub) : make_uint4(0, 0, 0, 0);
    }
    float acc[G][U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      float kf[VEC];
      unpack(v[i], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a = fmaf(qf[g][e], kf[e], a);
        acc[g][i] = a;
      }
    }
    // Sum over the LPR lanes of each row group.
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < U; ++i) acc[g][i] += __shfl_xor_sync(0xffffffffu, acc[g][i], off);

    // Lane `sub` of the group owns row i == sub.
    const int j = base + sub * NG + grp;
    if (sub < U && j < j_end) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < U; ++i)
          if (i == sub) s = acc[g][i];
        s *= scale;
        logits[(size_t)(b * Hq + hk * G + g) * ldn + j] = s;
        const float m_new = fmaxf(m_run[g], s);
        l_run[g] = l_run[g] * __expf(m_run[g] - m_new) + __expf(s - m_new);
        m_run[g] = m_new;
      }
    }
  }

  // CTA-wide merge of the (max, sum) pairs of each head.
  __shared__ float2 red[G][kScoreWarps];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float2 p = make_float2(m_run[g], l_run[g]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float2 o;
      o.x = __shfl_xor_sync(0xffffffffu, p.x, off);
      o.y = __shfl_xor_sync(0xffffffffu, p.y, off);
      p = lse_merge(p, o);
    }
    if (lane == 0) red[g][warp] = p;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float2 p = red[g][0];
#pragma unroll
    for (int w = 1; w < kScoreWarps; ++w) p = lse_merge(p, red[g][w]);
    part[(size_t)(u * G + g) * nchunks + c] = p;
  }
}

template <typename T, int D, int G>
cudaError_t launch_typed(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, cudaStream_t st) {
  const float scale = 1.0f / sqrtf((float)d.d);
  const unsigned grid = (unsigned)d.U * (unsigned)d.nchunks;
  score_kernel<T, D, G><<<grid, kScoreThreads, 0, st>>>(
      static_cast<const uint4*>(q_spec), static_cast<const uint4*>(k_dev), logits, part, d.n,
      d.ldn, d.Hq, d.Hkv, d.nchunks, scale);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_g(const Dims& d, const void* q, const void* k, float* lg, float2* p,
                     cudaStream_t st) {
  switch (d.G) {
    case 1: return launch_typed<T, D, 1>(d, q, k, lg, p, st);
    case 2: return launch_typed<T, D, 2>(d, q, k, lg, p, st);
    case 4: return launch_typed<T, D, 4>(d, q, k, lg, p, st);
    case 8: return launch_typed<T, D, 8>(d, q, k, lg, p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int score_chunk(int dtype, int head_dim) {
  if (dtype == DD_BF16) {
    if (head_dim == 64) return ScoreGeom<bf16_t, 64>::kChunk;
    if (head_dim == 128) return ScoreGeom<bf16_t, 128>::kChunk;
    if (head_dim == 256) return ScoreGeom<bf16_t, 256>::kChunk;
  } else {
    if (head_dim == 64) return ScoreGeom<float, 64>::kChunk;
    if (head_dim == 128) return ScoreGeom<float, 128>::kChunk;
  }
  return 0;
}

cudaError_t launch_score(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, cudaStream_t st) {
  if (d.dtype == DD_BF16) {
    if (d.d == 64) return launch_g<bf16_t, 64>(d, q_spec, k_dev, logits, part, st);
    if (d.d == 128) return launch_g<bf16_t, 128>(d, q_spec, k_dev, logits, part, st);
    if (d.d == 256) return launch_g<bf16_t, 256>(d, q_spec, k_dev, logits, part, st);
  } else {
    if (d.d == 64) return launch_g<float, 64>(d, q_spec, k_dev, logits, part, st);
    if (d.d == 128) return launch_g<float, 128>(d, q_spec, k_dev, logits, part, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
