// Step 4 of the decode step: decode attention of the real query over the
// gathered rows plus the local window,
//   o[b,h] = sum_{j in S} softmax_S(q[b,h] . K_j / sqrt(d)) V_j,
//   S = the k gathered rows followed by the W most recent positions.
// (DualDecoder paper Fig. 1 "Attention" over the gathered sparse KV; Sec. 2.1:
// attention of the current query over cached key/value entries.)
//
// Split-k: the k + W rows of a unit are cut into splits of 64 rows; one CTA
// per (split, unit) computes, for every query head of the group, the partial
// (max m, sum l of exp(e - m), o = sum exp(e - m) V) so that each K/V row is
// read once per group.  A second, tiny kernel merges the splits with the
// log-sum-exp rule o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
#include <math.h>

#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int RS = kAttnRowsPerSplit;

template <typename T, int D>
struct AttnGeom {
  static constexpr int kVec = Elem<T>::kVec;
  static constexpr int kLpr = D / kVec;
  static constexpr int kRpw = 32 / kLpr;
  static constexpr int kGroups = kAttnWarps * kRpw;  // row groups per CTA
  static constexpr int kIt = RS / kGroups;           // rows per group per split
  static_assert(RS % kGroups == 0, "split must be a multiple of the row groups");
};

// The log-sum-exp merge of one output element over the nsplit partials of
// its (request, query head) row; `CG` reads partials written by other CTAs of
// the same launch past L1.
template <bool CG>
__device__ __forceinline__ float merge_splits(const float* part_o, const float2* part_ml,
                                              size_t row, int nsplit, int D, int t) {
  const float2* ml = part_ml + row * nsplit;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, (CG ? __ldcg(ml + s) : ml[s]).x);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float2 v = CG ? __ldcg(ml + s) : ml[s];
    const float w = __expf(v.x - M);
    L = fmaf(w, v.y, L);
    const float* po = part_o + (row * nsplit + s) * D + t;
    acc = fmaf(w, CG ? __ldcg(po) : *po, acc);
  }
  return acc / L;
}

// MERGE: the last split CTA of each unit to finish (per-unit counters, zero
// before the launch and after it) also merges the unit's G output rows, so no
// separate merge launch is needed.
template <typename T, int D, int G, bool MERGE>
__global__ void __launch_bounds__(kAttnThreads)
    attn_partial_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k_buf,
                        const uint4* __restrict__ v_buf, const uint4* __restrict__ k_win,
                        const uint4* __restrict__ v_win, float* __restrict__ part_o,
                        float2* __restrict__ part_ml, int kw_stride, int kw_off, int k, int W,
                        int Hq, int Hkv, int nsplit, float scale, int32_t* __restrict__ counters,
                        float* __restrict__ out) {
  using Geo = AttnGeom<T, D>;
  constexpr int VEC = Geo::kVec, LPR = Geo::kLpr, RPW = Geo::kRpw, NG = Geo::kGroups;
  constexpr int IT = Geo::kIt, V16 = LPR;

  const int u = blockIdx.x, s = blockIdx.y;
  const int b = u / Hkv, hk = u - b * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPR, grp = warp * RPW + lane / LPR;
  const int R = k + W, r0 = s * RS, nr = min(R, r0 + RS) - r0;

  __shared__ float e_sh[G][RS];
  __shared__ float2 ml_sh[G];
  __shared__ float o_sh[NG][G][D];

  float qf[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g) unpack(ld_ro(q + (size_t)(b * Hq + hk * G + g) * V16 + sub), qf[g]);

  // Row r of the unit's attended set: gathered row r (r < k) or window row
  // r - k, i.e. cached position n - W + (r - k): row kw_off + (r - k) of the
  // unit's kw_stride rows of k_win (the key cache: stride n, offset n - W; a
  // window buffer: stride W, offset 0).
  auto k_row = [&](int r) -> const uint4* {
    return (r < k) ? k_buf + ((size_t)u * k + r) * V16
                   : k_win + ((size_t)u * kw_stride + kw_off + (r - k)) * V16;
  };
  auto v_row = [&](int r) -> const uint4* {
    return (r < k) ? v_buf + ((size_t)u * k + r) * V16 : v_win + ((size_t)u * W + (r - k)) * V16;
  };

  // Both the K and the V rows of this lane are requested up front, so the
  // softmax below does not wait for a second round trip to memory.
  uint4 vv[IT];
  // Phase 1: logits of this split's rows.
  {
    uint4 kv[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      const int rl = i * NG + grp;
      kv[i] = (rl < nr) ? ld_ro(k_row(r0 + rl) + sub) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      const int rl = i * NG + grp;
      vv[i] = (rl < nr) ? ld_ro(v_row(r0 + rl) + sub) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      float kf[VEC];
      unpack(kv[i], kf);
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a = fmaf(qf[g][e], kf[e], a);
        acc[g] = a;
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], off);
      const int rl = i * NG + grp;
      if (sub == 0 && rl < nr) {
#pragma unroll
        for (int g = 0; g < G; ++g) e_sh[g][rl] = acc[g] * scale;
      }
    }
  }
  __syncthreads();

  // Phase 2: per head, m = max e, p = exp(e - m), l = sum p.
  for (int g = warp; g < G; g += kAttnWarps) {
    float m = -INFINITY;
    for (int r = lane; r < nr; r += 32) m = fmaxf(m, e_sh[g][r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int r = lane; r < nr; r += 32) {
      const float p = __expf(e_sh[g][r] - m);
      e_sh[g][r] = p;
      l += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) ml_sh[g] = make_float2(m, l);
  }
  __syncthreads();

  // Phase 3: o = sum_r p_r V_r, rows split over the row groups.
  float acc[G][VEC];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
  {
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      const int rl = i * NG + grp;
      if (rl < nr) {
        float vf[VEC];
        unpack(vv[i], vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = e_sh[g][rl];
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < VEC; ++e) o_sh[grp][g][sub * VEC + e] = acc[g][e];
  __syncthreads();

  for (int x = threadIdx.x; x < G * D; x += kAttnThreads) {
    const int g = x / D, t = x - g * D;
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < NG; ++r) sum += o_sh[r][g][t];
    part_o[((size_t)(u * G + g) * nsplit + s) * D + t] = sum;
  }
  if (threadIdx.x < G) part_ml[(size_t)(u * G + threadIdx.x) * nsplit + s] = ml_sh[threadIdx.x];
  if (!MERGE) return;

  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(counters + u, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) counters[u] = 0;  // ready for the next launch
  for (int x = threadIdx.x; x < G * D; x += kAttnThreads) {
    const int g = x / D, t = x - g * D;
    const size_t row = (size_t)u * G + g;  // = b H_q + h_kv G + g
    out[row * D + t] = merge_splits<true>(part_o, part_ml, row, nsplit, D, t);
  }
}

// One CTA of D threads per (request, query head): log-sum-exp merge of the splits.
__global__ void attn_merge_kernel(const float* __restrict__ part_o,
                                  const float2* __restrict__ part_ml, float* __restrict__ out,
                                  int nsplit, int D) {
  const int row = blockIdx.x, t = threadIdx.x;
  out[(size_t)row * D + t] = merge_splits<false>(part_o, part_ml, row, nsplit, D, t);
}

template <typename T, int D, int G>
cudaError_t launch_typed(const Dims& d, const void* q, const void* kb, const void* vb,
                         const WindowK& kw, const void* vw, float* out, float* po, float2* pml,
                         int32_t* counters, cudaStream_t st) {
  static unsigned long long prepared = 0, prepared_fused = 0, prepared_merge = 0;
  const float scale = 1.0f / sqrtf((float)d.d);
  const dim3 grid((unsigned)d.U, (unsigned)d.nsplit);
  if (counters) {  // partials and merge in one launch
    cudaError_t e0 = prepare_kernel(attn_partial_kernel<T, D, G, true>, &prepared_fused, 0);
    if (e0 != cudaSuccess) return e0;
    attn_partial_kernel<T, D, G, true><<<grid, kAttnThreads, 0, st>>>(
        static_cast<const uint4*>(q), static_cast<const uint4*>(kb),
        static_cast<const uint4*>(vb), static_cast<const uint4*>(kw.p),
        static_cast<const uint4*>(vw), po, pml, kw.stride, kw.off, d.k, d.W, d.Hq, d.Hkv,
        d.nsplit, scale, counters, out);
    return cudaGetLastError();
  }
  cudaError_t e0 = prepare_kernel(attn_partial_kernel<T, D, G, false>, &prepared, 0);
  if (e0 == cudaSuccess) e0 = prepare_kernel(attn_merge_kernel, &prepared_merge, 0);
  if (e0 != cudaSuccess) return e0;
  attn_partial_kernel<T, D, G, false><<<grid, kAttnThreads, 0, st>>>(
      static_cast<const uint4*>(q), static_cast<const uint4*>(kb), static_cast<const uint4*>(vb),
      static_cast<const uint4*>(kw.p), static_cast<const uint4*>(vw), po, pml, kw.stride, kw.off,
      d.k, d.W, d.Hq, d.Hkv, d.nsplit, scale, nullptr, nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_merge_kernel<<<(unsigned)(d.B * d.Hq), D, 0, st>>>(po, pml, out, d.nsplit, D);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_g(const Dims& d, const void* q, const void* kb, const void* vb,
                     const WindowK& kd, const void* vw, float* out, float* po, float2* pml,
                     int32_t* cnt, cudaStream_t st) {
  switch (d.G) {
    case 1: return launch_typed<T, D, 1>(d, q, kb, vb, kd, vw, out, po, pml, cnt, st);
    case 2: return launch_typed<T, D, 2>(d, q, kb, vb, kd, vw, out, po, pml, cnt, st);
    case 4: return launch_typed<T, D, 4>(d, q, kb, vb, kd, vw, out, po, pml, cnt, st);
    case 8: return launch_typed<T, D, 8>(d, q, kb, vb, kd, vw, out, po, pml, cnt, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attn(const Dims& d, const void* q, const void* k_buf, const void* v_buf,
                        const WindowK& k_dev, const void* v_win, float* out, float* part_o,
                        float2* part_ml, cudaStream_t st, int32_t* counters) {
  if (d.dtype == DD_BF16) {
    if (d.d == 64) return launch_g<bf16_t, 64>(d, q, k_buf, v_buf, k_dev, v_win, out, part_o, part_ml, counters, st);
    if (d.d == 128) return launch_g<bf16_t, 128>(d, q, k_buf, v_buf, k_dev, v_win, out, part_o, part_ml, counters, st);
    if (d.d == 256) return launch_g<bf16_t, 256>(d, q, k_buf, v_buf, k_dev, v_win, out, part_o, part_ml, counters, st);
  } else {
    if (d.d == 64) return launch_g<float, 64>(d, q, k_buf, v_buf, k_dev, v_win, out, part_o, part_ml, counters, st);
    if (d.d == 128) return launch_g<float, 128>(d, q, k_buf, v_buf, k_dev, v_win, out, part_o, part_ml, counters, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
