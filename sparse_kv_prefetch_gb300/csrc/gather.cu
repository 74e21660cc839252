// Step 3 of the decode step: gather the selected K/V rows from the pinned
// host-memory KV store into the layer-scoped GPU buffer.  (DualDecoder paper,
// Sec. 2.2 and Fig. 1 "Sparse KV Gather": the selected entries are scattered
// over the context, so they are gathered from host memory across the
// host-to-device link; summary page worked example, step 5.)
//
// The SMs read host memory directly (zero-copy: page-locked memory is mapped
// into the GPU's unified address space), so the scattered rows never need a
// host-side gather or one copy-engine request per row.  Consecutive threads
// read consecutive 16-byte pieces of a row (a row of d elements is d*elt/16
// pieces; K and V pieces of the same row are adjacent), and every thread keeps
// kInFlight independent host loads outstanding to cover the link latency.
// The grid is small on purpose: it must leave room for the scoring kernel
// that runs concurrently on the compute stream.
#include "dd_internal.cuh"

namespace dd {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kInFlight = 8;

template <int CPR>  // 16-byte pieces per row
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint4* __restrict__ k_host, const uint4* __restrict__ v_host,
                  const int32_t* __restrict__ idx, uint4* __restrict__ k_buf,
                  uint4* __restrict__ v_buf, int n, int k, long long rows) {
  // Piece p of the flattened work list: row r = p / (2 CPR), tensor t (K or
  // V) = (p / CPR) & 1, part = p % CPR.
  const long long total = rows * 2 * CPR;
  const long long stride = (long long)gridDim.x * kGatherThreads;
  for (long long p0 = (long long)blockIdx.x * kGatherThreads + threadIdx.x; p0 < total;
       p0 += stride * kInFlight) {
    uint4 v[kInFlight];
    long long dst[kInFlight];
    int tv[kInFlight];
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      const long long p = p0 + i * stride;
      tv[i] = -1;
      if (p < total) {
        const unsigned r = (unsigned)(p / (2 * CPR));
        const int t = (int)((p / CPR) & 1);
        const int part = (int)(p % CPR);
        const unsigned u = r / (unsigned)k;
        const int j = min(max(__ldg(idx + r), 0), n - 1);  // never read outside the store
        const uint4* src = (t ? v_host : k_host) + (((long long)u * n + j) * CPR + part);
        v[i] = ld_ro(src);
        dst[i] = (long long)r * CPR + part;
        tv[i] = t;
      }
    }
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      if (tv[i] == 0) k_buf[dst[i]] = v[i];
      if (tv[i] == 1) v_buf[dst[i]] = v[i];
    }
  }
}

template <int CPR>
cudaError_t launch_typed(const Dims& d, const void* kh, const void* vh, const int32_t* idx,
                         void* kb, void* vb, cudaStream_t st) {
  const long long rows = (long long)d.U * d.k;
  const long long work = (rows * 2 * CPR + (long long)kGatherThreads * kInFlight - 1) /
                         ((long long)kGatherThreads * kInFlight);
  long long grid = sm_count();  // one CTA per SM at most
  if (grid > work) grid = work;
  if (grid < 1) grid = 1;
  gather_kernel<CPR><<<(unsigned)grid, kGatherThreads, 0, st>>>(
      static_cast<const uint4*>(kh), static_cast<const uint4*>(vh), idx,
      static_cast<uint4*>(kb), static_cast<uint4*>(vb), d.n, d.k, rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const Dims& d, const void* k_host, const void* v_host,
                          const int32_t* idx, void* k_buf, void* v_buf, cudaStream_t st) {
  switch (d.d * d.elt / 16) {
    case 8: return launch_typed<8>(d, k_host, v_host, idx, k_buf, v_buf, st);
    case 16: return launch_typed<16>(d, k_host, v_host, idx, k_buf, v_buf, st);
    case 32: return launch_typed<32>(d, k_host, v_host, idx, k_buf, v_buf, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
