// Step 2 of the decode step: per (request, KV head) top-k of the selection
// score, I = argtopk(a, k) over positions [0, n - W), ties to the lower
// position, written in ascending position order.  (DualDecoder summary page,
// core formulas: I = argtopk(alpha, k); paper Fig. 1 "Select Top-k".)
//
// The selection score is a[j] = exp(s_j - LSE) for MHA; since exp is
// monotone the kernel ranks the fp32 logits themselves.  For grouped-query
// heads a[j] = sum over the group of exp(s_hj - LSE_h) in fp32.  LSE_h is
// first merged from the scoring kernel's per-chunk (max, sum) pairs.
//
// Exact radix select on order-preserving 32-bit keys, one CTA per unit.  Each
// warp owns a contiguous segment of the positions, so position order is the
// order (warp, position within the warp's segment):
//   pass A  histogram of key bits 31..21 over the unit (global reads); the
//           bucket b1 that holds the k-th largest key is found by a block
//           scan from the top;
//   pass B  every warp compacts the keys of its segment with top bits >= b1,
//           in position order, into its own shared-memory list (ballots and
//           shuffle scans only, no block barrier);
//   refine  bits 20..10 and 9..0 of the threshold key T are resolved on the
//           lists with two more histograms;
//   emit    every key > T plus the first (lowest-position) k_rem keys equal
//           to T are written; each warp places its entries after the counts of
//           the warps before it.
// If a warp's list would overflow (very many near-equal scores), the refine
// and emit steps run over global memory instead: the same result.
#include <math.h>

#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kPer = 4;                   // consecutive positions per lane per step
constexpr int kWarpStep = 32 * kPer;      // positions per warp per step
constexpr int kTile = kTkThreads * kPer;  // positions per block-wide step (fallback)
constexpr int kWarpCap = 512;             // list entries per warp
constexpr int kListCap = kWarpCap * kTkWarps;

struct TkSmem {
  uint32_t hist[2048];
  uint32_t wt[32];
  uint32_t res[2];
  uint32_t wcnt[kTkWarps];  // list entries per warp
  uint32_t wgt[kTkWarps];   // per warp: entries > T, then their exclusive prefix
  uint32_t weq[kTkWarps];   // per warp: entries == T, then their exclusive prefix
  uint32_t overflow;
  float lse[8];
  uint32_t keys[kListCap];
  int32_t idxs[kListCap];
};

// Order-preserving map float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, int lane) {
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  return x - v;
}

// Exclusive prefix sum of v over the block in thread order; *total = sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wt, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wt[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kTkWarps ? wt[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    if (lane < kTkWarps) wt[lane] = t;
  }
  __syncthreads();
  const uint32_t r = (warp ? wt[warp - 1] : 0u) + x - v;
  *total = wt[kTkWarps - 1];
  __syncthreads();
  return r;
}

// Given a complete histogram, find the bin b with
//   above(b) < k_rem <= above(b) + hist[b],  above(b) = sum_{x > b} hist[x],
// and store (b, above(b)) in res.  Requires 1 <= k_rem <= sum(hist).
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t k_rem, uint32_t* wt,
                         uint32_t* res) {
  const int per = nbins / kTkThreads;  // bins per thread, top bins first
  const int top = nbins - 1 - (int)threadIdx.x * per;
  uint32_t local = 0;
  for (int p = 0; p < per; ++p) local += hist[top - p];
  uint32_t tot;
  const uint32_t excl = block_excl_scan(local, wt, &tot);
  if (excl < k_rem && k_rem <= excl + local) {
    uint32_t acc = excl;
    for (int p = 0; p < per; ++p) {
      const uint32_t h = hist[top - p];
      if (acc + h >= k_rem) {
        res[0] = (uint32_t)(top - p);
        res[1] = acc;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

// Keys of one unit computed from the fp32 logits in global memory.
template <int G>
struct GlobalKeys {
  const float* lg;  // logits row of the group's first query head
  int ldn, span;
  float lse[G];
  // Keys of positions j0..j0+3 (j0 % 4 == 0, j0 < span); entries >= span
  // hold unspecified values and must be masked by the caller.
  __device__ __forceinline__ void load4(int j0, uint32_t (&key)[kPer]) const {
    if (G == 1) {
      const float4 v = *reinterpret_cast<const float4*>(lg + j0);
      key[0] = f2key(v.x);
      key[1] = f2key(v.y);
      key[2] = f2key(v.z);
      key[3] = f2key(v.w);
    } else {
      float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 v = *reinterpret_cast<const float4*>(lg + (size_t)g * ldn + j0);
        a[0] += __expf(v.x - lse[g]);
        a[1] += __expf(v.y - lse[g]);
        a[2] += __expf(v.z - lse[g]);
        a[3] += __expf(v.w - lse[g]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) key[e] = f2key(a[e]);
    }
  }
};

// Histogram over the whole unit (block-strided) of bits [lo, lo+nbits) of the
// keys whose higher bits equal `prefix`.
template <int G>
__device__ void histogram_global(const GlobalKeys<G>& src, TkSmem& sm, int lo, int nbits,
                                 uint32_t prefix) {
  const int nb = 1 << nbits;
  for (int i = threadIdx.x; i < nb; i += kTkThreads) sm.hist[i] = 0;
  __syncthreads();
  for (int j0 = (int)threadIdx.x * kPer; j0 < src.span; j0 += kTile) {
    uint32_t key[kPer];
    src.load4(j0, key);
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (j0 + e < src.span && (key[e] >> (lo + nbits)) == prefix)
        atomicAdd(&sm.hist[(key[e] >> lo) & (uint32_t)(nb - 1)], 1u);
  }
  __syncthreads();
}

// Histogram over the per-warp lists (each warp walks its own list).
__device__ void histogram_lists(TkSmem& sm, int lo, int nbits, uint32_t prefix) {
  const int nb = 1 << nbits;
  for (int i = threadIdx.x; i < nb; i += kTkThreads) sm.hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* keys = sm.keys + warp * kWarpCap;
  const int cnt = (int)sm.wcnt[warp];
  for (int e = lane; e < cnt; e += 32) {
    const uint32_t key = keys[e];
    if ((key >> (lo + nbits)) == prefix) atomicAdd(&sm.hist[(key >> lo) & (uint32_t)(nb - 1)], 1u);
  }
  __syncthreads();
}

// Score written for a selected key: alpha (MHA) or the group score itself.
__device__ __forceinline__ float sel_value(uint32_t key, bool mha, float lse0) {
  const float v = key2f(key);
  return mha ? expf(v - lse0) : v;
}

// Ordered emit over the per-warp lists: every key > T, then the first k_rem
// keys == T in position order.
__device__ void emit_lists(TkSmem& sm, uint32_t T, uint32_t k_rem, int k, int32_t* idx_out,
                           float* sel_out, bool mha, float lse0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* keys = sm.keys + warp * kWarpCap;
  const int32_t* idxs = sm.idxs + warp * kWarpCap;
  const int cnt = (int)sm.wcnt[warp];
  uint32_t ngt = 0, neq = 0;
  for (int e = lane; e < cnt; e += 32) {
    ngt += keys[e] > T;
    neq += keys[e] == T;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ngt += __shfl_xor_sync(0xffffffffu, ngt, off);
    neq += __shfl_xor_sync(0xffffffffu, neq, off);
  }
  if (lane == 0) {
    sm.wgt[warp] = ngt;
    sm.weq[warp] = neq;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t g = lane < kTkWarps ? sm.wgt[lane] : 0u;
    const uint32_t q = lane < kTkWarps ? sm.weq[lane] : 0u;
    const uint32_t gx = warp_excl_scan(g, lane), qx = warp_excl_scan(q, lane);
    if (lane < kTkWarps) {
      sm.wgt[lane] = gx;
      sm.weq[lane] = qx;
    }
  }
  __syncthreads();
  uint32_t gb = sm.wgt[warp], eb = sm.weq[warp];  // counts before this warp's segment
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int e0 = 0; e0 < cnt; e0 += 32) {
    const int e = e0 + lane;
    const bool v = e < cnt;
    const uint32_t key = v ? keys[e] : 0u;
    const bool gt = v && key > T, eq = v && key == T;
    const unsigned bg = __ballot_sync(0xffffffffu, gt), bq = __ballot_sync(0xffffffffu, eq);
    const uint32_t g_before = gb + __popc(bg & lt_mask), q_before = eb + __popc(bq & lt_mask);
    int pos = -1;
    if (gt) pos = (int)(g_before + min(q_before, k_rem));
    else if (eq && q_before < k_rem) pos = (int)(g_before + q_before);
    if (pos >= 0 && pos < k) {
      idx_out[pos] = idxs[e];
      sel_out[pos] = sel_value(key, mha, lse0);
    }
    gb += __popc(bg);
    eb += __popc(bq);
  }
}

// Ordered emit over global memory (fallback), block-wide in tiles.
template <int G>
__device__ void emit_global(const GlobalKeys<G>& src, TkSmem& sm, uint32_t T, uint32_t k_rem,
                            int k, int32_t* idx_out, float* sel_out, bool mha, float lse0) {
  uint32_t cgt = 0, ceq = 0;
  for (int t0 = 0; t0 < src.span; t0 += kTile) {
    const int j0 = t0 + (int)threadIdx.x * kPer;
    uint32_t key[kPer] = {0u, 0u, 0u, 0u};
    if (j0 < src.span) src.load4(j0, key);
    bool gt[kPer], eq[kPer];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const bool v = j0 + e < src.span;
      gt[e] = v && key[e] > T;
      eq[e] = v && key[e] == T;
      ngt += gt[e];
      neq += eq[e];
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan(ngt | (neq << 16), sm.wt, &tot);
    uint32_t gb = cgt + (ex & 0xFFFFu), eb = ceq + (ex >> 16);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      int pos = -1;
      if (gt[e]) {
        pos = (int)(gb + min(eb, k_rem));
        ++gb;
      } else if (eq[e]) {
        if (eb < k_rem) pos = (int)(gb + eb);
        ++eb;
      }
      if (pos >= 0 && pos < k) {
        idx_out[pos] = j0 + e;
        sel_out[pos] = sel_value(key[e], mha, lse0);
      }
    }
    cgt += tot & 0xFFFFu;
    ceq += tot >> 16;
  }
}

template <int G>
__global__ void __launch_bounds__(kTkThreads)
    topk_kernel(const float* __restrict__ logits, const float2* __restrict__ part,
                int32_t* __restrict__ idx_out, float* __restrict__ sel_out,
                float* __restrict__ lse_out, int Hq, int Hkv, int ldn, int span, int k,
                int nchunks) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TkSmem& sm = *reinterpret_cast<TkSmem*>(smem_raw);
  const int u = blockIdx.x, b = u / Hkv, hk = u - b * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // LSE of each query head of the group from the per-chunk (max, sum) pairs.
  if (warp < G) {
    const float2* pp = part + (size_t)(u * G + warp) * nchunks;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int c = lane; c < nchunks; c += 32) acc = lse_merge(acc, pp[c]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float2 o;
      o.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
      o.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc = lse_merge(acc, o);
    }
    if (lane == 0) {
      const float lse = acc.x + logf(acc.y);
      sm.lse[warp] = lse;
      if (lse_out) lse_out[b * Hq + hk * G + warp] = lse;
    }
  }
  if (threadIdx.x == 0) sm.overflow = 0;
  for (int i = threadIdx.x; i < 2048; i += kTkThreads) sm.hist[i] = 0;
  __syncthreads();

  GlobalKeys<G> src;
  src.lg = logits + (size_t)(b * Hq + hk * G) * ldn;
  src.ldn = ldn;
  src.span = span;
#pragma unroll
  for (int g = 0; g < G; ++g) src.lse[g] = sm.lse[g];
  int32_t* idx_u = idx_out + (size_t)u * k;
  float* sel_u = sel_out + (size_t)u * k;

  // This warp's segment of positions: [seg0, seg1), seg0 a multiple of 4.
  const int per_warp =
      ((span + kTkWarps - 1) / kTkWarps + kWarpStep - 1) / kWarpStep * kWarpStep;
  const int seg0 = min(span, warp * per_warp), seg1 = min(span, seg0 + per_warp);

  // Pass A: bucket of the k-th largest key by its top 11 bits.
  for (int j0 = seg0 + lane * kPer; j0 < seg1; j0 += kWarpStep) {
    uint32_t key[kPer];
    src.load4(j0, key);
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (j0 + e < seg1) atomicAdd(&sm.hist[key[e] >> 21], 1u);
  }
  __syncthreads();
  find_bin(sm.hist, 2048, (uint32_t)k, sm.wt, sm.res);
  const uint32_t b1 = sm.res[0];
  uint32_t k_rem = (uint32_t)k - sm.res[1];
  __syncthreads();

  // Pass B: each warp compacts its keys in buckets >= b1, in position order.
  {
    uint32_t* keys = sm.keys + warp * kWarpCap;
    int32_t* idxs = sm.idxs + warp * kWarpCap;
    uint32_t n_w = 0;
    bool over = false;
    for (int base = seg0; base < seg1; base += kWarpStep) {
      const int j0 = base + lane * kPer;
      uint32_t key[kPer] = {0u, 0u, 0u, 0u};
      if (j0 < seg1) src.load4(j0, key);
      bool f[kPer];
      uint32_t c = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        f[e] = (j0 + e < seg1) && (key[e] >> 21) >= b1;
        c += f[e];
      }
      uint32_t pos = n_w + warp_excl_scan(c, lane);
      uint32_t tot = c;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
      if (n_w + tot > (uint32_t)kWarpCap) {
        over = true;  // the same decision in every lane
        break;
      }
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        if (f[e]) {
          keys[pos] = key[e];
          idxs[pos] = j0 + e;
          ++pos;
        }
      }
      n_w += tot;
    }
    if (lane == 0) {
      sm.wcnt[warp] = n_w;
      if (over) atomicOr(&sm.overflow, 1u);
    }
  }
  __syncthreads();

  uint32_t T;
  if (!sm.overflow) {
    histogram_lists(sm, 10, 11, b1);
    find_bin(sm.hist, 2048, k_rem, sm.wt, sm.res);
    const uint32_t pre = (b1 << 11) | sm.res[0];
    k_rem -= sm.res[1];
    __syncthreads();
    histogram_lists(sm, 0, 10, pre);
    find_bin(sm.hist, 1024, k_rem, sm.wt, sm.res);
    T = (pre << 10) | sm.res[0];
    k_rem -= sm.res[1];
    __syncthreads();
    emit_lists(sm, T, k_rem, k, idx_u, sel_u, G == 1, sm.lse[0]);
  } else {
    // A warp list overflowed: resolve the remaining bits and emit from global memory.
    histogram_global(src, sm, 10, 11, b1);
    find_bin(sm.hist, 2048, k_rem, sm.wt, sm.res);
    const uint32_t pre = (b1 << 11) | sm.res[0];
    k_rem -= sm.res[1];
    __syncthreads();
    histogram_global(src, sm, 0, 10, pre);
    find_bin(sm.hist, 1024, k_rem, sm.wt, sm.res);
    T = (pre << 10) | sm.res[0];
    k_rem -= sm.res[1];
    __syncthreads();
    emit_global(src, sm, T, k_rem, k, idx_u, sel_u, G == 1, sm.lse[0]);
  }
}

template <int G>
cudaError_t launch_typed(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                         float* sel, float* lse, cudaStream_t st) {
  static unsigned long long prepared = 0;
  cudaError_t e = prepare_kernel(topk_kernel<G>, &prepared, (int)sizeof(TkSmem));
  if (e != cudaSuccess) return e;
  topk_kernel<G><<<d.U, kTkThreads, sizeof(TkSmem), st>>>(logits, part, idx, sel, lse, d.Hq,
                                                          d.Hkv, d.ldn, d.span, d.k, d.nchunks);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                        float* sel, float* lse, cudaStream_t st) {
  switch (d.G) {
    case 1: return launch_typed<1>(d, logits, part, idx, sel, lse, st);
    case 2: return launch_typed<2>(d, logits, part, idx, sel, lse, st);
    case 4: return launch_typed<4>(d, logits, part, idx, sel, lse, st);
    case 8: return launch_typed<8>(d, logits, part, idx, sel, lse, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
