// Internal declarations shared by the kernels and the C-ABI layer of libdd.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

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
  size_t logits, part, attn_o, attn_ml, sel_true, counters, attn_counters, total;
};

dd_status resolve(const dd_shape* s, Dims* out);
WsLayout ws_layout(const Dims& d);

constexpr int kAttnRowsPerSplit = 64;

// Kernel launchers (score.cu, topk.cu, gather.cu, attn.cu).  Each returns the
// launch status (cudaGetLastError after the launch).
cudaError_t launch_score(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, cudaStream_t st);
// With expand = c > 1 each selected position j is written as the c rows
// j c .. j c + c - 1 (idx is then [U][k c]); sel stays [U][k].
cudaError_t launch_topk(const Dims& d, const float* logits, const float2* part, int32_t* idx,
                        float* sel, float* lse, cudaStream_t st, int expand = 1);
// Scoring of fp32 keys (landmarks, d.dtype == DD_F32) by a bf16 query.
cudaError_t launch_score_bf16_query(const Dims& d, const void* q_bf16, const void* k_f32,
                                    float* logits, float2* part, cudaStream_t st);
// Scoring with the selection fused in: the last CTA of each unit runs its
// top-k.  counters [U] must be zero before the launch and are zero after it.
cudaError_t launch_score_select(const Dims& d, const void* q_spec, const void* k_dev,
                                float* logits, float2* part, int32_t* counters, int32_t* idx,
                                float* sel, float* lse, cudaStream_t st);
// Where the host store's rows are, as device-accessible addresses: position j
// of unit u has its K row at k + (u n + j) hs and its V row at v + (u n + j) hs
// bytes.  hs is the row's bytes for separate K and V stores; for one store
// holding each position's K row followed by its V row, v = k + row bytes and
// hs = twice the row bytes.
struct HostKV {
  const void* k;
  const void* v;
  size_t hs;
};
// touch: first read one word per huge page of the host stores (worth it only
// for stores backed by huge pages, i.e. from dd_host_alloc).
cudaError_t launch_gather(const Dims& d, const HostKV& h, const int32_t* idx, void* k_buf,
                          void* v_buf, int mode, cudaStream_t st, bool touch);
// Geometry of the bulk-copy gather (mode 0), process-wide: grid in percent
// of the SM count, bytes per tensor of a shared-memory stage, stages per CTA.
dd_status set_gather_geometry(int grid_pct, int tile_bytes, int stages);
// The same for the load/store gather (mode 1): grid in percent of the SM
// count, threads per CTA (a multiple of 32, at most 256).
dd_status set_gather_lsu_geometry(int grid_pct, int threads);
// Host stores allocated by the library (hoststore.cu).
// True if p lies in a store from dd_host_alloc (transparent huge pages,
// registered with CUDA), whose translations the gather prefetches.
bool in_huge_page_store(const void* p);
// Device-accessible address of page-locked host memory known to CUDA (a
// host KV store); NULL otherwise.
const void* host_to_device(const void* p);

// Pointer checks of the C ABI (api.cu): device memory of the current device,
// or managed memory; all_device accepts NULL entries.
bool is_device_ptr(const void* p);
// The load/store gather (mode 1) indexes 16-byte pieces with 31 bits: the
// gathered rows of one tensor must stay below 8 GiB.
bool lsu_gather_fits(const Dims& d);
bool all_device(std::initializer_list<const void*> ps);
// Where the attention reads the window's keys: row off + i (i < W) of each
// unit's `stride` rows starting at p.
struct WindowK {
  const void* p;
  int stride, off;
};
// The window inside the key cache [U][n][d], or a window buffer [U][W][d].
inline WindowK window_in_cache(const void* k_dev, const Dims& d) {
  return WindowK{k_dev, d.n, d.n - d.W};
}
inline WindowK window_buffer(const void* k_win, const Dims& d) { return WindowK{k_win, d.W, 0}; }

// With counters ([U], zero before the launch and after it) the merge of the
// splits runs inside the partial kernel (one launch); without, as a second
// kernel.
cudaError_t launch_attn(const Dims& d, const void* q, const void* k_buf, const void* v_buf,
                        const WindowK& k_win, const void* v_win, float* out, float* part_o,
                        float2* part_ml, cudaStream_t st, int32_t* counters = nullptr);

// Miss correction (correct.cu): copy each row of the real query's top-k from
// the prefetched buffer, or from the host store where the prediction missed.
constexpr int kMaxCorrectK = 4096;
cudaError_t launch_fixup(const Dims& d, const int32_t* idx_spec, const int32_t* idx_true,
                         const float* sel_true, const void* kb_spec, const void* vb_spec,
                         const HostKV& h, void* kb_out, void* vb_out, int32_t* miss_out,
                         float* mass_out, cudaStream_t st);

// Landmark selection (landmark.cu).
cudaError_t launch_landmarks(const Dims& d, int chunk, const void* k_dev, float* landmarks,
                             cudaStream_t st);
cudaError_t launch_expand(const int32_t* chunks, int32_t* rows, int units, int kc, int chunk,
                          cudaStream_t st);
cudaError_t launch_to_f32(const void* x_bf16, float* y, int count, cudaStream_t st);

// Shapes of landmark selection: `full` is the layer, `lm` the landmark "key
// cache" (M = (n - W) / chunk rows of fp32, k / chunk to select, no window).
// Workspace offsets of the fp32 queries and the selected chunk ids follow
// lm's own layout.
struct LandmarkDims {
  Dims full, lm;
  WsLayout lay;
  size_t q32, chunks, total;
  int chunk;
};
dd_status resolve_landmarks(const dd_shape* s, int chunk, LandmarkDims* out);

// Number of kernels each launcher enqueues.
// (The gather is 2 launches with the huge-page touch, 1 without.)
// (Attention is 1 launch in the layer loop, whose workspace keeps merge counters.)
constexpr int kScoreLaunches = 1, kTopkLaunches = 1, kGatherLaunches = 2, kAttnLaunches = 2,
              kFixupLaunches = 1, kScoreSelectLaunches = 1;

// Steps 1-2 of one layer into idx / sel / lse, with the workspace laid out by
// `lay`: the fused kernel (counters at lay.counters must be zero) or, if
// !fused, the scoring and top-k kernels.  Adds the kernels launched to
// *launches.
cudaError_t select_rows(const Dims& d, const WsLayout& lay, char* ws, const void* q,
                        const void* k_dev, int32_t* idx, float* sel, float* lse, bool fused,
                        cudaStream_t st, int* launches);

// Huge-page size of the host (transparent huge pages), read once; 2 MiB if
// the host does not report one.  Host stores from dd_host_alloc use it.
size_t host_page_bytes();

int sm_count();

// Once per device and kernel: opt in to `dyn_smem` bytes of dynamic shared
// memory (if above the default 48 KB) and ask for the largest shared-memory
// carveout.  Every kernel of the library asks for the same carveout, so the
// SMs never need a different L1/shared split to host kernels of the compute
// and copy streams side by side.
template <typename Kernel>
cudaError_t prepare_kernel(Kernel* fn, unsigned long long* done_mask, int dyn_smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  if (dyn_smem > 48 * 1024) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
  return cudaSuccess;
}

// Keys per scoring CTA for a stored dtype, head size, number of units and
// keys per unit (0 if the dtype or head size is unsupported).
int score_chunk(int dtype, int head_dim, long long units, int n);

// Whether the scoring kernel computes this stored dtype and group size (query
// heads per KV head) on the tensor cores rather than in the per-lane form.
bool score_uses_mma(int dtype, int group);

// Read and clear the device-side status words that kernels set when a bounded
// wait gives up (nonzero: some wait timed out since the last read).
unsigned int take_score_status();
unsigned int take_gather_status();
unsigned int take_debug_status();

// Test hooks (debug.cu): a bounded GPU sleep on a stream, and a wait that
// nothing completes, which gives up after limit_ns and sets the status word.
cudaError_t launch_delay(uint64_t ns, cudaStream_t st);
cudaError_t launch_expire_wait(uint64_t limit_ns, cudaStream_t st);

// ----------------------------------------------------------------- device

// log2 of a power of two, at compile time.
__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

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

// ------------------------------------------------ async copies (TMA, mbarrier)
//
// Bulk copies (cp.async.bulk) move contiguous byte ranges between global and
// shared memory on the SM's tensor-memory-access unit, without occupying the
// load/store pipeline; completion is signalled on an mbarrier in shared memory
// through its transaction count.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// Make the initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that lets the thread sleep up to hint_ns while the phase is
// incomplete (it consumes no issue slots meanwhile).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Every wait in this library is bounded: after kWaitLimitNs the wait gives up
// and returns false; the caller records DD_ERR_TIMEOUT and stops its work.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}
// mbar_wait for long waits (host-memory copies): sleeps between polls.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity,
                                                uint32_t hint_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity, hint_ns))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
// global -> shared, completion counted on `bar` (bytes and addresses 16-aligned).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// An L2 policy that evicts the lines it tags first (for data read once).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_load with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gmem_src,
                                               uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// shared -> global, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until the committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Merge two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(m, a.y * __expf(a.x - m) + b.y * __expf(b.x - m));
}

}  // namespace dd
