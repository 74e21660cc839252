// Miss correction on the critical path.  The rows prefetched for a layer were
// selected with the speculated token's query; once the real query is known,
// its own top-k is computed (the same scoring and selection kernels), and the
// attention must use exactly those rows.  Every true row that the prediction
// already brought to the GPU is copied from the prefetched buffer; every row
// it missed is fetched from the host store now.  (DualDecoder paper, Sec. 1:
// the layer-aware transfer schedule "corrects prediction misses on the
// critical path"; summary page, weaknesses: mispredictions fall back to
// synchronous retrieval.)  The counts of missed rows and the share of the true
// top-k's probability mass that the prediction covered are the predictability
// measurements of the paper's Sec. 1 claim.
//
// fixup_kernel: one CTA per (request, KV head).  Each true position is looked
// up in the ascending prefetched list by binary search; the per-slot source
// (prefetched slot, or host position) goes to shared memory; then the CTA
// copies the rows, 16 bytes per thread and several pieces in flight.
#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kFixThreads = 256;
constexpr int kFixInFlight = 4;

template <int CPR>  // 16-byte pieces per row
__global__ void __launch_bounds__(kFixThreads)
    fixup_kernel(const int32_t* __restrict__ idx_spec, const int32_t* __restrict__ idx_true,
                 const float* __restrict__ sel_true, const uint4* __restrict__ kb_spec,
                 const uint4* __restrict__ vb_spec, const uint4* __restrict__ k_host,
                 const uint4* __restrict__ v_host, uint4* __restrict__ kb_out,
                 uint4* __restrict__ vb_out, int32_t* __restrict__ miss_out,
                 float* __restrict__ mass_out, int n, int k, int hsp) {
  extern __shared__ int32_t src[];  // slot of the prefetched buffer, or -(1 + host position)
  __shared__ int red_i[kFixThreads / 32];
  __shared__ float red_h[kFixThreads / 32], red_a[kFixThreads / 32];
  const int u = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t* is = idx_spec + (size_t)u * k;
  const int32_t* it = idx_true + (size_t)u * k;

  int misses = 0;
  float hit_mass = 0.f, all_mass = 0.f;
  for (int i = threadIdx.x; i < k; i += kFixThreads) {
    const int j = __ldg(it + i);
    int lo = 0, hi = k;  // first slot with is[slot] >= j
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(is + mid) < j) lo = mid + 1;
      else hi = mid;
    }
    const bool hit = lo < k && __ldg(is + lo) == j;
    src[i] = hit ? lo : -(1 + j);
    const float a = __ldg(sel_true + (size_t)u * k + i);
    all_mass += a;
    if (hit) hit_mass += a;
    else ++misses;
  }
  __syncthreads();

  const int total = k * 2 * CPR;  // piece p: slot p / (2 CPR), tensor (p / CPR) & 1
  for (int p0 = threadIdx.x; p0 < total; p0 += kFixThreads * kFixInFlight) {
    uint4 v[kFixInFlight];
#pragma unroll
    for (int r = 0; r < kFixInFlight; ++r) {
      const int p = p0 + r * kFixThreads;
      if (p < total) {
        const int i = p / (2 * CPR), t = (p / CPR) & 1, part = p % CPR;
        const int s = src[i];
        if (s >= 0) {
          v[r] = ld_ro((t ? vb_spec : kb_spec) + ((size_t)u * k + s) * CPR + part);
        } else {
          const int j = min(max(-s - 1, 0), n - 1);  // never outside the store
          v[r] = ld_ro((t ? v_host : k_host) + ((size_t)u * n + j) * hsp + part);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kFixInFlight; ++r) {
      const int p = p0 + r * kFixThreads;
      if (p < total) {
        const int i = p / (2 * CPR), t = (p / CPR) & 1, part = p % CPR;
        (t ? vb_out : kb_out)[((size_t)u * k + i) * CPR + part] = v[r];
      }
    }
  }

#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    misses += __shfl_xor_sync(0xffffffffu, misses, off);
    hit_mass += __shfl_xor_sync(0xffffffffu, hit_mass, off);
    all_mass += __shfl_xor_sync(0xffffffffu, all_mass, off);
  }
  if (lane == 0) {
    red_i[warp] = misses;
    red_h[warp] = hit_mass;
    red_a[warp] = all_mass;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    float h = 0.f, a = 0.f;
    for (int w = 0; w < kFixThreads / 32; ++w) {
      m += red_i[w];
      h += red_h[w];
      a += red_a[w];
    }
    if (miss_out) miss_out[u] = m;
    if (mass_out) {
      mass_out[2 * (size_t)u] = h;
      mass_out[2 * (size_t)u + 1] = a;
    }
  }
}

template <int CPR>
cudaError_t launch_fix(const Dims& d, const int32_t* idx_spec, const int32_t* idx_true,
                       const float* sel_true, const void* kb_spec, const void* vb_spec,
                       const HostKV& h, void* kb_out, void* vb_out, int32_t* miss_out,
                       float* mass_out, cudaStream_t st) {
  static unsigned long long prepared = 0;
  const int smem = d.k * (int)sizeof(int32_t);
  cudaError_t e = prepare_kernel(fixup_kernel<CPR>, &prepared, kMaxCorrectK * (int)sizeof(int32_t));
  if (e != cudaSuccess) return e;
  fixup_kernel<CPR><<<d.U, kFixThreads, smem, st>>>(
      idx_spec, idx_true, sel_true, static_cast<const uint4*>(kb_spec),
      static_cast<const uint4*>(vb_spec), static_cast<const uint4*>(h.k),
      static_cast<const uint4*>(h.v), static_cast<uint4*>(kb_out), static_cast<uint4*>(vb_out),
      miss_out, mass_out, d.n, d.k, (int)(h.hs / 16));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fixup(const Dims& d, const int32_t* idx_spec, const int32_t* idx_true,
                         const float* sel_true, const void* kb_spec, const void* vb_spec,
                         const HostKV& h, void* kb_out, void* vb_out, int32_t* miss_out,
                         float* mass_out, cudaStream_t st) {
  switch (d.d * d.elt / 16) {
    case 8: return launch_fix<8>(d, idx_spec, idx_true, sel_true, kb_spec, vb_spec, h, kb_out, vb_out, miss_out, mass_out, st);
    case 16: return launch_fix<16>(d, idx_spec, idx_true, sel_true, kb_spec, vb_spec, h, kb_out, vb_out, miss_out, mass_out, st);
    case 32: return launch_fix<32>(d, idx_spec, idx_true, sel_true, kb_spec, vb_spec, h, kb_out, vb_out, miss_out, mass_out, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
