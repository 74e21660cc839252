// Step 2 of the decode step as its own kernel: per (request, KV head) top-k
// of the selection score over positions [0, n - W), ties to the lower
// position, written in ascending position order.  One 512-thread CTA per
// unit runs the exact radix selection of select.cuh after merging the LSE of
// every query head of its group from the scoring kernel's per-chunk (max,
// sum) pairs.  This is the default form of step 2; with DD_STEP_FUSED_TOPK
// the scoring kernel (score.cu) runs the same selection in its last CTA of
// each unit instead.
#include "select.cuh"

namespace dd {
namespace {

constexpr int kTkWarps = 16;
constexpr int kTkThreads = kTkWarps * 32;
constexpr int kWarpCap = 512;  // list entries per warp
using TkSmem = sel::Smem<kTkWarps, kWarpCap>;

template <int G>
__global__ void __launch_bounds__(kTkThreads)
    topk_kernel(const float* __restrict__ logits, const float2* __restrict__ part,
                int32_t* __restrict__ idx_out, float* __restrict__ sel_out,
                float* __restrict__ lse_out, int Hq, int Hkv, int ldn, int span, int k,
                int nchunks, int expand) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TkSmem& sm = *reinterpret_cast<TkSmem*>(smem_raw);
  const int u = blockIdx.x, b = u / Hkv, hk = u - b * Hkv;
  sel::merge_lse<G, false>(part, u, b, hk, Hq, nchunks, lse_out, sm);
  sel::sync<kTkWarps>();
  sel::select_unit<G, false>(sm, logits + (size_t)(b * Hq + hk * G) * ldn, ldn, span, k,
                             idx_out + (size_t)u * k * expand, sel_out + (size_t)u * k, expand);
}

template <int G>
cudaError_t launch_typed(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                         float* sel, float* lse, int expand, cudaStream_t st) {
  static unsigned long long prepared = 0;
  cudaError_t e = prepare_kernel(topk_kernel<G>, &prepared, (int)sizeof(TkSmem));
  if (e != cudaSuccess) return e;
  topk_kernel<G><<<d.U, kTkThreads, sizeof(TkSmem), st>>>(
      logits, part, idx, sel, lse, d.Hq, d.Hkv, d.ldn, d.span, d.k, d.nchunks, expand);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                        float* sel, float* lse, cudaStream_t st, int expand) {
  switch (d.G) {
    case 1: return launch_typed<1>(d, logits, part, idx, sel, lse, expand, st);
    case 2: return launch_typed<2>(d, logits, part, idx, sel, lse, expand, st);
    case 4: return launch_typed<4>(d, logits, part, idx, sel, lse, expand, st);
    case 8: return launch_typed<8>(d, logits, part, idx, sel, lse, expand, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dd
