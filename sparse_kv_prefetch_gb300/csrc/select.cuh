// Exact per-unit top-k selection (step 2 of the decode step), as device code
// shared by the standalone top-k kernel (topk.cu, one 512-thread CTA per
// unit) and the fused scoring kernel (score.cu, whose last CTA of a unit runs
// the selection with its eight consumer warps).
//
// The selection score is a[j] = exp(s_j - LSE) for MHA; since exp is monotone
// the fp32 logits themselves are ranked.  For grouped-query heads a[j] = sum
// over the group of exp(s_hj - LSE_h) in fp32.  (DualDecoder summary page,
// core formulas: I = argtopk(alpha, k); paper Fig. 1 "Select Top-k".)
//
// Exact radix select on order-preserving 32-bit keys.  Each warp owns a
// contiguous segment of the positions, so position order is the order
// (warp, position within the warp's segment):
//   sample  (n - W >= 16384) a histogram of one 128-position block in 16 sets
//           a bucket b_low expected to keep ~1.5 k keys; one full pass B with
//           b_low, and if it kept >= k keys without overflowing a list, b1 is
//           found on the lists and pass A is skipped; else the exact passes:
//   pass A  histogram of key bits 31..21 over the unit; the bucket b1 that
//           holds the k-th largest key is found by a block scan from the top;
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
//
// Barriers are the named barrier 1 over the WARPS selecting warps, so a CTA
// with more warps (the fused kernel's producer warp) can leave them out.
#pragma once

#include <math.h>

#include "dd_internal.cuh"

namespace dd {
namespace sel {

constexpr int kPer = 4;                // consecutive positions per lane per load
constexpr int kWarpStep = 32 * kPer;  // positions per warp per load
constexpr int kUnroll = 4;            // loads in flight per lane in passes A and B
constexpr int kSampleEvery = 16;      // the sample: one warp step in 16
constexpr int kSampleMin = 16384;     // positions below which no sample is taken

template <int WARPS, int WCAP>
struct Smem {
  uint32_t hist[2048];
  uint32_t wt[32];
  uint32_t res[2];
  uint32_t wcnt[WARPS];  // list entries per warp
  uint32_t wgt[WARPS];   // per warp: entries > T, then their exclusive prefix
  uint32_t weq[WARPS];   // per warp: entries == T, then their exclusive prefix
  uint32_t overflow;
  uint32_t nsample;  // positions in the sample (sampled threshold)
  float lse[8];
  uint32_t keys[WCAP * WARPS];
  int32_t idxs[WCAP * WARPS];
};

template <int WARPS>
__device__ __forceinline__ void sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
}

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

// Exclusive prefix sum of v over the selecting threads in thread order;
// *total = sum.
template <int WARPS>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wt, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wt[warp] = x;
  sync<WARPS>();
  if (warp == 0) {
    uint32_t t = lane < WARPS ? wt[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    if (lane < WARPS) wt[lane] = t;
  }
  sync<WARPS>();
  const uint32_t r = (warp ? wt[warp - 1] : 0u) + x - v;
  *total = wt[WARPS - 1];
  sync<WARPS>();
  return r;
}

// Given a complete histogram, find the bin b with
//   above(b) < k_rem <= above(b) + hist[b],  above(b) = sum_{x > b} hist[x],
// and store (b, above(b)) in res.  Requires 1 <= k_rem <= sum(hist).
template <int WARPS>
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t k_rem, uint32_t* wt,
                         uint32_t* res) {
  const int per = nbins / (WARPS * 32);  // bins per thread, top bins first
  const int top = nbins - 1 - (int)threadIdx.x * per;
  uint32_t local = 0;
  for (int p = 0; p < per; ++p) local += hist[top - p];
  uint32_t tot;
  const uint32_t excl = block_excl_scan<WARPS>(local, wt, &tot);
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
  sync<WARPS>();
}

// Keys of one unit computed from the fp32 logits in global memory.  With CG
// the loads bypass L1 (the logits were written by other CTAs of the same
// launch).
template <int G, bool CG>
struct GlobalKeys {
  const float* lg;  // logits row of the group's first query head
  int ldn, span;
  float lse[G];
  __device__ __forceinline__ float4 ld4(const float* p) const {
    return CG ? __ldcg(reinterpret_cast<const float4*>(p))
              : *reinterpret_cast<const float4*>(p);
  }
  // Keys of positions j0..j0+3 (j0 % 4 == 0, j0 < span); entries >= span
  // hold unspecified values and must be masked by the caller.
  __device__ __forceinline__ void load4(int j0, uint32_t (&key)[kPer]) const {
    if (G == 1) {
      const float4 v = ld4(lg + j0);
      key[0] = f2key(v.x);
      key[1] = f2key(v.y);
      key[2] = f2key(v.z);
      key[3] = f2key(v.w);
    } else {
      float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 v = ld4(lg + (size_t)g * ldn + j0);
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

// Histogram over the whole unit (strided over the selecting threads) of bits
// [lo, lo+nbits) of the keys whose higher bits equal `prefix`.
template <int WARPS, int WCAP, int G, bool CG>
__device__ void histogram_global(const GlobalKeys<G, CG>& src, Smem<WARPS, WCAP>& sm, int lo,
                                 int nbits, uint32_t prefix) {
  constexpr int kTile = WARPS * 32 * kPer;
  const int nb = 1 << nbits;
  for (int i = threadIdx.x; i < nb; i += WARPS * 32) sm.hist[i] = 0;
  sync<WARPS>();
  for (int j0 = (int)threadIdx.x * kPer; j0 < src.span; j0 += kTile) {
    uint32_t key[kPer];
    src.load4(j0, key);
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (j0 + e < src.span && (key[e] >> (lo + nbits)) == prefix)
        atomicAdd(&sm.hist[(key[e] >> lo) & (uint32_t)(nb - 1)], 1u);
  }
  sync<WARPS>();
}

// Histogram over the per-warp lists (each warp walks its own list).
template <int WARPS, int WCAP>
__device__ void histogram_lists(Smem<WARPS, WCAP>& sm, int lo, int nbits, uint32_t prefix) {
  const int nb = 1 << nbits;
  for (int i = threadIdx.x; i < nb; i += WARPS * 32) sm.hist[i] = 0;
  sync<WARPS>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* keys = sm.keys + warp * WCAP;
  const int cnt = (int)sm.wcnt[warp];
  for (int e = lane; e < cnt; e += 32) {
    const uint32_t key = keys[e];
    if ((key >> (lo + nbits)) == prefix) atomicAdd(&sm.hist[(key >> lo) & (uint32_t)(nb - 1)], 1u);
  }
  sync<WARPS>();
}

// Index written for a selected position j: j itself, or with expand = c > 1
// (landmark selection, where j is a chunk) the c rows j c .. j c + c - 1 of
// the chunk, at slots pos c .. pos c + c - 1.
__device__ __forceinline__ void put_index(int32_t* idx_out, int pos, int j, int expand) {
  if (expand == 1) {
    idx_out[pos] = j;
  } else {
    for (int r = 0; r < expand; ++r) idx_out[pos * expand + r] = j * expand + r;
  }
}

// Score written for a selected key: alpha (MHA) or the group score itself.
__device__ __forceinline__ float sel_value(uint32_t key, bool mha, float lse0) {
  const float v = key2f(key);
  return mha ? expf(v - lse0) : v;
}

// Ordered emit over the per-warp lists: every key > T, then the first k_rem
// keys == T in position order.
template <int WARPS, int WCAP>
__device__ void emit_lists(Smem<WARPS, WCAP>& sm, uint32_t T, uint32_t k_rem, int k,
                           int32_t* idx_out, float* sel_out, bool mha, float lse0, int expand) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* keys = sm.keys + warp * WCAP;
  const int32_t* idxs = sm.idxs + warp * WCAP;
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
  sync<WARPS>();
  if (warp == 0) {
    const uint32_t g = lane < WARPS ? sm.wgt[lane] : 0u;
    const uint32_t q = lane < WARPS ? sm.weq[lane] : 0u;
    const uint32_t gx = warp_excl_scan(g, lane), qx = warp_excl_scan(q, lane);
    if (lane < WARPS) {
      sm.wgt[lane] = gx;
      sm.weq[lane] = qx;
    }
  }
  sync<WARPS>();
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
      put_index(idx_out, pos, idxs[e], expand);
      sel_out[pos] = sel_value(key, mha, lse0);
    }
    gb += __popc(bg);
    eb += __popc(bq);
  }
}

// Ordered emit over global memory (fallback), in tiles over the selecting threads.
template <int WARPS, int WCAP, int G, bool CG>
__device__ void emit_global(const GlobalKeys<G, CG>& src, Smem<WARPS, WCAP>& sm, uint32_t T,
                            uint32_t k_rem, int k, int32_t* idx_out, float* sel_out, bool mha,
                            float lse0, int expand) {
  constexpr int kTile = WARPS * 32 * kPer;
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
    const uint32_t ex = block_excl_scan<WARPS>(ngt | (neq << 16), sm.wt, &tot);
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
        put_index(idx_out, pos, j0 + e, expand);
        sel_out[pos] = sel_value(key[e], mha, lse0);
      }
    }
    cgt += tot & 0xFFFFu;
    ceq += tot >> 16;
  }
}

// LSE of each query head of unit u's group from the per-chunk (max, sum)
// pairs, into sm.lse (and lse_out if not NULL).  Warps 0..G-1 work; the
// caller synchronises afterwards.
template <int G, bool CG, int WARPS, int WCAP>
__device__ void merge_lse(const float2* part, int u, int b, int hk, int Hq, int nchunks,
                          float* lse_out, Smem<WARPS, WCAP>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < G) {
    const float2* pp = part + (size_t)(u * G + warp) * nchunks;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int c = lane; c < nchunks; c += 32)
      acc = lse_merge(acc, CG ? __ldcg(pp + c) : pp[c]);
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
}

// The whole selection of one unit, with sm.lse already set and visible to
// the selecting threads: k positions of [0, span) into idx_u (ascending;
// each expanded to `expand` consecutive rows, see put_index) and their
// selection scores into sel_u.
template <int G, bool CG, int WARPS, int WCAP>
__device__ void select_unit(Smem<WARPS, WCAP>& sm, const float* lg, int ldn, int span, int k,
                            int32_t* idx_u, float* sel_u, int expand = 1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) sm.overflow = 0;
  for (int i = threadIdx.x; i < 2048; i += WARPS * 32) sm.hist[i] = 0;
  sync<WARPS>();

  GlobalKeys<G, CG> src;
  src.lg = lg;
  src.ldn = ldn;
  src.span = span;
#pragma unroll
  for (int g = 0; g < G; ++g) src.lse[g] = sm.lse[g];

  // This warp's segment of positions: [seg0, seg1), seg0 a multiple of 4.
  const int per_warp = ((span + WARPS - 1) / WARPS + kWarpStep - 1) / kWarpStep * kWarpStep;
  const int seg0 = min(span, warp * per_warp), seg1 = min(span, seg0 + per_warp);

  // Pass A: histogram of the top 11 key bits over the whole unit.  Each lane
  // issues kUnroll loads before using any (memory-level parallelism).
  auto pass_a = [&]() {
    for (int base = seg0; base < seg1; base += kWarpStep * kUnroll) {
      uint32_t key[kUnroll][kPer];
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep + lane * kPer;
        if (j0 < seg1) src.load4(j0, key[v]);
      }
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
          if (j0 + e < seg1) atomicAdd(&sm.hist[key[v][e] >> 21], 1u);
      }
    }
    sync<WARPS>();
  };

  // Pass B: each warp compacts its keys whose top bits are >= thr, in
  // position order, into its own shared-memory list.
  auto pass_b = [&](uint32_t thr) {
    uint32_t* keys = sm.keys + warp * WCAP;
    int32_t* idxs = sm.idxs + warp * WCAP;
    uint32_t n_w = 0;
    bool over = false;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = seg0; base < seg1 && !over; base += kWarpStep * kUnroll) {
      uint32_t key[kUnroll][kPer];
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep + lane * kPer;
        if (j0 < seg1) src.load4(j0, key[v]);
      }
      // The kUnroll groups in position order: group v covers
      // [base + v kWarpStep, base + (v + 1) kWarpStep).
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep + lane * kPer;
        bool f[kPer];
        unsigned bal[kPer];
        unsigned any = 0;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          f[e] = (j0 + e < seg1) && (key[v][e] >> 21) >= thr;
          bal[e] = __ballot_sync(0xffffffffu, f[e]);
          any |= bal[e];
        }
        if (!any) continue;  // most steps: no candidate in the warp
        // Position order is (lane, e): the entries of the lanes before this
        // one come first, then this lane's in e order.
        uint32_t tot = 0, pos = n_w;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          tot += __popc(bal[e]);
          pos += __popc(bal[e] & lt_mask);
        }
        if (n_w + tot > (uint32_t)WCAP) {
          over = true;  // the same decision in every lane
          break;
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          if (f[e]) {
            keys[pos] = key[v][e];
            idxs[pos] = j0 + e;
            ++pos;
          }
        }
        n_w += tot;
      }
    }
    if (lane == 0) {
      sm.wcnt[warp] = n_w;
      if (over) atomicOr(&sm.overflow, 1u);
    }
    sync<WARPS>();
  };

  uint32_t b1 = 0, k_rem = 0;
  bool ready = false;  // lists hold every key of bucket >= b1; b1, k_rem exact
  if (span >= kSampleMin) {
    // Sampled threshold: a histogram of one warp step in kSampleEvery gives a
    // bucket b_low that keeps about 1.5 times the expected number of top-k
    // keys above it; one full pass compacts every key of bucket >= b_low.  If
    // that holds at least k keys (so all of the top k) and no list overflowed,
    // the exact bucket b1 comes from the lists alone: one pass over the
    // logits instead of two.  Otherwise the exact two passes run.
    if (threadIdx.x == 0) sm.nsample = 0;
    sync<WARPS>();
    uint32_t mine = 0;
    for (int base = seg0; base < seg1; base += kWarpStep * kSampleEvery * kUnroll) {
      uint32_t key[kUnroll][kPer];
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep * kSampleEvery + lane * kPer;
        if (j0 < seg1) src.load4(j0, key[v]);
      }
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        const int j0 = base + v * kWarpStep * kSampleEvery + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
          if (j0 + e < seg1) {
            atomicAdd(&sm.hist[key[v][e] >> 21], 1u);
            ++mine;
          }
      }
    }
    if (mine) atomicAdd(&sm.nsample, mine);
    sync<WARPS>();
    const uint32_t ns = sm.nsample;
    const uint32_t ks = (uint32_t)(((unsigned long long)k * ns * 3) / (2ull * span)) + 8;
    if (ks <= ns) {
      find_bin<WARPS>(sm.hist, 2048, ks, sm.wt, sm.res);
      const uint32_t b_low = sm.res[0];
      sync<WARPS>();
      pass_b(b_low);
      uint32_t cand = 0;
      for (int w = 0; w < WARPS; ++w) cand += sm.wcnt[w];
      if (!sm.overflow && cand >= (uint32_t)k) {
        // Exact b1 and the count above it, from the candidates.
        for (int i = threadIdx.x; i < 2048; i += WARPS * 32) sm.hist[i] = 0;
        sync<WARPS>();
        {
          const uint32_t* keys = sm.keys + warp * WCAP;
          const int cnt = (int)sm.wcnt[warp];
          for (int e = lane; e < cnt; e += 32) atomicAdd(&sm.hist[keys[e] >> 21], 1u);
        }
        sync<WARPS>();
        find_bin<WARPS>(sm.hist, 2048, (uint32_t)k, sm.wt, sm.res);
        b1 = sm.res[0];
        k_rem = (uint32_t)k - sm.res[1];
        ready = true;
      }
      sync<WARPS>();
    }
    if (!ready) {
      if (threadIdx.x == 0) sm.overflow = 0;
      for (int i = threadIdx.x; i < 2048; i += WARPS * 32) sm.hist[i] = 0;
      sync<WARPS>();
    }
  }
  if (!ready) {
    pass_a();
    find_bin<WARPS>(sm.hist, 2048, (uint32_t)k, sm.wt, sm.res);
    b1 = sm.res[0];
    k_rem = (uint32_t)k - sm.res[1];
    sync<WARPS>();
    pass_b(b1);
  }

  uint32_t T;
  if (!sm.overflow) {
    histogram_lists(sm, 10, 11, b1);
    find_bin<WARPS>(sm.hist, 2048, k_rem, sm.wt, sm.res);
    const uint32_t pre = (b1 << 11) | sm.res[0];
    k_rem -= sm.res[1];
    sync<WARPS>();
    histogram_lists(sm, 0, 10, pre);
    find_bin<WARPS>(sm.hist, 1024, k_rem, sm.wt, sm.res);
    T = (pre << 10) | sm.res[0];
    k_rem -= sm.res[1];
    sync<WARPS>();
    emit_lists(sm, T, k_rem, k, idx_u, sel_u, G == 1, sm.lse[0], expand);
  } else {
    // A warp list overflowed: resolve the remaining bits and emit from global memory.
    histogram_global(src, sm, 10, 11, b1);
    find_bin<WARPS>(sm.hist, 2048, k_rem, sm.wt, sm.res);
    const uint32_t pre = (b1 << 11) | sm.res[0];
    k_rem -= sm.res[1];
    sync<WARPS>();
    histogram_global(src, sm, 0, 10, pre);
    find_bin<WARPS>(sm.hist, 1024, k_rem, sm.wt, sm.res);
    T = (pre << 10) | sm.res[0];
    k_rem -= sm.res[1];
    sync<WARPS>();
    emit_global(src, sm, T, k_rem, k, idx_u, sel_u, G == 1, sm.lse[0], expand);
  }
}

}  // namespace sel
}  // namespace dd
