// Step 3 of the decode step: gather the selected K/V rows from the pinned
// host-memory KV store into the layer-scoped GPU buffer.  (DualDecoder paper,
// Sec. 2.2 and Fig. 1 "Sparse KV Gather": the selected entries are scattered
// over the context, so they are gathered from host memory across the
// host-to-device link; summary page worked example, step 5.)
//
// The GPU reads host memory directly (zero-copy: page-locked memory is
// mapped into its unified address space), so the scattered rows never need a
// host-side gather or one copy-engine request per row.  Two kernels:
//
// mode 0, gather_tma_kernel: each CTA is one warp that moves tiles of R
//   consecutive selected rows of one (request, KV head).  Its lanes issue one
//   bulk copy (cp.async.bulk, executed by the SM's tensor-memory-access unit)
//   per K row and per V row, from host memory into a shared-memory stage; the
//   stage completes on an mbarrier and is written to the scratch buffer with
//   two contiguous bulk stores.  Several stages stay in flight per CTA.  The
//   load/store pipeline is never blocked on the long host-link latency.  The
//   kernel is built to run beside the scoring kernel of the next layer: by
//   default one CTA per SM, small enough to fit next to three scoring CTAs;
//   host lines tagged L2 evict-first; the waiting lane sleeps between polls.
//   (Measured on GB300: a grid of two 64 KiB CTAs per SM took CTA slots
//   from the scoring kernel and hid 17 % of the gather on the GQA-128K
//   layer; the small geometry hides 64-76 %.)
//
// mode 1, gather_lsu_kernel: every thread keeps kInFlight 16-byte loads from
//   host memory outstanding (consecutive threads read consecutive 16-byte
//   pieces of a row) through the load/store pipeline.
#include <algorithm>
#include <atomic>

#include "dd_internal.cuh"

namespace dd {
namespace {

__device__ unsigned int g_gather_status = 0;

// ---------------------------------------------------- translation prefetch
//
// The GPU reaches host memory through the host's page tables.  When thousands
// of gather requests first hit a page whose translation is not cached, every
// one of them waits on the same translation, and the storm also delays the
// other kernels' memory requests.  Before each gather one warp therefore reads
// one word per huge page of the layer's K and V regions (at the region start
// and at every page boundary inside it, so every read stays inside the
// caller's buffer): each translation is then resolved once, and the gather
// that follows runs at full speed.  With huge pages (dd_host_alloc) this is a
// handful of reads per layer.
__global__ void __launch_bounds__(32)
    touch_pages_kernel(const unsigned char* __restrict__ k_host,
                       const unsigned char* __restrict__ v_host, size_t bytes, size_t stride,
                       unsigned int* __restrict__ sink) {
  unsigned int acc = 0;
  for (int t = 0; t < 2; ++t) {
    const unsigned char* base = t ? v_host : k_host;
    const uintptr_t start = (uintptr_t)base, end = start + bytes;
    const uintptr_t first = (start / stride + 1) * stride;  // first page boundary after start
    const size_t n_pages = end > first ? (end - first + stride - 1) / stride : 0;
    for (size_t i = threadIdx.x; i <= n_pages; i += 32) {
      const uintptr_t a = i == 0 ? start : first + (i - 1) * stride;
      if (a < end) acc += *reinterpret_cast<const volatile unsigned int*>(a & ~(uintptr_t)3);
    }
  }
  if (acc == 0x9E3779B9u) *sink = acc;  // keeps the reads; practically never taken
}

__device__ unsigned int g_touch_sink = 0;

// ------------------------------------------------------------ mode 0 (TMA)
//
// Geometry of a launch: `ctas` one-warp CTAs, each with `stages` shared-memory
// stages of R rows per tensor (R = tile bytes / row bytes).  Rows in flight
// are ctas * stages * R per tensor; the default (one CTA per SM, 3 stages of
// 4 KiB) needs 24 KiB of shared memory per CTA, which fits beside three
// scoring CTAs on an SM.  dd_set_gather_geometry changes it process-wide.
constexpr int kMaxStages = 8;
// A stage waits on the host link for microseconds: the waiting lane sleeps up
// to this long between polls instead of taking issue slots from the kernels
// running beside the gather on the same SM.
constexpr uint32_t kWaitSleepNs = 2000;
constexpr int kMaxTileBytes = 16384;
constexpr int kMaxDynSmem = 227 * 1024;  // largest opt-in per CTA
std::atomic<int> g_grid_pct{100}, g_tile_bytes{4096}, g_stages{3};

size_t tma_smem(int rows, int rb, int stages) {
  return (size_t)2 * stages * rows * rb + (size_t)stages * sizeof(uint64_t);
}

template <int RB>  // bytes per row
__global__ void __launch_bounds__(32)
    gather_tma_kernel(const unsigned char* __restrict__ k_host,
                      const unsigned char* __restrict__ v_host, const int32_t* __restrict__ idx,
                      unsigned char* __restrict__ k_buf, unsigned char* __restrict__ v_buf, int n,
                      int k, int units, int R, int stages, size_t hs) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tile_bytes = R * RB;
  const bool runs = hs == RB;  // consecutive positions are contiguous in the store
  unsigned char* ring_k = smem;
  unsigned char* ring_v = smem + (size_t)stages * tile_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)2 * stages * tile_bytes);
  const int lane = threadIdx.x;
  const int tiles_per_unit = (k + R - 1) / R;
  const int n_tiles = units * tiles_per_unit;

  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncwarp();

  // Issue the row copies of `tile` into stage s.  Rows whose positions are
  // consecutive (whole chunks under landmark selection) are contiguous in a
  // store of separate K and V rows and in the tile, so each run of them is
  // one bulk copy: the lane holding the first row of a run copies the run.
  auto issue = [&](int tile, int s) {
    const int u = tile / tiles_per_unit, i0 = (tile - u * tiles_per_unit) * R;
    const int nr = min(R, k - i0);
    if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * nr * RB));
    __syncwarp();
    for (int r0 = 0; r0 < nr; r0 += 32) {
      const int r = r0 + lane;
      const bool valid = r < nr;
      int j = 0;
      if (valid) j = min(max(__ldg(idx + (size_t)u * k + i0 + r), 0), n - 1);  // never outside
      const int jp = __shfl_up_sync(0xffffffffu, j, 1);
      const bool cont = runs && valid && lane > 0 && jp + 1 == j;  // continues the run before it
      const unsigned cmask = __ballot_sync(0xffffffffu, cont);
      if (valid && !cont) {
        const unsigned after = lane == 31 ? 0u : cmask >> (lane + 1);
        const int len = __ffs(~after);  // this row plus the continuing rows after it
        const size_t src = ((size_t)u * n + j) * hs;
        const uint32_t bytes = (uint32_t)(len * RB);
        // Host lines are read once: evict them first, so they do not push the
        // scoring kernel's logits out of L2.
        const uint64_t pol = l2_evict_first_policy();
        bulk_load_hint(ring_k + (size_t)s * tile_bytes + (size_t)r * RB, k_host + src, bytes,
                       &full[s], pol);
        bulk_load_hint(ring_v + (size_t)s * tile_bytes + (size_t)r * RB, v_host + src, bytes,
                       &full[s], pol);
      }
    }
  };

  for (int p = 0; p < stages; ++p) {
    const int t = blockIdx.x + p * gridDim.x;
    if (t < n_tiles) issue(t, p);
  }
  bool ok = true;
  int it = 0;
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
    const int s = it % stages;
    if (!mbar_wait_sleep(&full[s], (it / stages) & 1, kWaitSleepNs)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      const int u = t / tiles_per_unit, i0 = (t - u * tiles_per_unit) * R;
      const int nr = min(R, k - i0);
      const size_t dst = ((size_t)u * k + i0) * RB;
      bulk_store(k_buf + dst, ring_k + (size_t)s * tile_bytes, (uint32_t)(nr * RB));
      bulk_store(v_buf + dst, ring_v + (size_t)s * tile_bytes, (uint32_t)(nr * RB));
      bulk_commit();
      bulk_wait_read_all();  // the stage may be refilled once the stores have read it
    }
    __syncwarp();
    const int nt = t + stages * gridDim.x;
    if (nt < n_tiles) issue(nt, s);
  }
  if (!ok) {
    if (lane == 0) atomicOr(&g_gather_status, 1u);
    // let the copies still in flight land before the CTA exits
    for (int s = 0; s < stages; ++s) {
      mbar_wait(&full[s], 0);
      mbar_wait(&full[s], 1);
    }
  }
  if (lane == 0) bulk_wait_all();
}

template <int RB>
cudaError_t launch_tma(const Dims& d, const HostKV& h, const int32_t* idx, void* kb, void* vb,
                       cudaStream_t st) {
  static unsigned long long prepared = 0;
  cudaError_t e = prepare_kernel(gather_tma_kernel<RB>, &prepared, kMaxDynSmem);
  if (e != cudaSuccess) return e;
  const int R = std::max(1, std::min(64, g_tile_bytes.load() / RB));
  const int stages = g_stages.load();
  const long long tiles = (long long)d.U * ((d.k + R - 1) / R);
  long long grid = ((long long)sm_count() * g_grid_pct.load() + 99) / 100;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  gather_tma_kernel<RB><<<(unsigned)grid, 32, tma_smem(R, RB, stages), st>>>(
      static_cast<const unsigned char*>(h.k), static_cast<const unsigned char*>(h.v), idx,
      static_cast<unsigned char*>(kb), static_cast<unsigned char*>(vb), d.n, d.k, d.U, R,
      stages, h.hs);
  return cudaGetLastError();
}

// ------------------------------------------------------------ mode 1 (LSU)
// Geometry of a launch: `threads` per CTA (one to eight warps) and the grid
// in percent of the SM count, each thread with kInFlight 16-byte loads in
// flight; dd_set_gather_lsu_geometry changes it process-wide.  (One warp per
// SM with 16 loads in flight, small enough to sit beside the grouped-query
// scoring kernel, reached only 32-51 GB/s: too shallow for the host link.)
constexpr int kLsuMaxThreads = 256;
constexpr int kInFlight = 8;
std::atomic<int> g_lsu_grid_pct{100}, g_lsu_threads{kLsuMaxThreads};

template <int CPR, int INFL>  // 16-byte pieces per row, loads in flight per thread
__device__ __forceinline__ void gather_lsu_body(const uint4* __restrict__ k_host,
                                                const uint4* __restrict__ v_host,
                                                const int32_t* __restrict__ idx,
                                                uint4* __restrict__ k_buf,
                                                uint4* __restrict__ v_buf, int n, int k,
                                                long long rows, long long hsp) {
  // Piece p of the flattened work list: row r = p / (2 CPR), tensor t (K or
  // V) = (p / CPR) & 1, part = p % CPR.  Consecutive threads read consecutive
  // pieces of a row.  Host lines are read once: streaming loads.
  const long long total = rows * 2 * CPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; p0 < total;
       p0 += stride * INFL) {
    uint4 v[INFL];
    // Where each loaded piece goes: piece index into k_buf / v_buf, times 2,
    // plus the tensor (the launcher keeps 2 * total below 2^31); -1 if none.
    int dst[INFL];
#pragma unroll
    for (int i = 0; i < INFL; ++i) {
      const long long p = p0 + i * stride;
      dst[i] = -1;
      if (p < total) {
        const unsigned r = (unsigned)(p / (2 * CPR));
        const int t = (int)((p / CPR) & 1);
        const int part = (int)(p % CPR);
        const unsigned u = r / (unsigned)k;
        const int j = min(max(__ldg(idx + r), 0), n - 1);  // never read outside the store
        const uint4* src = (t ? v_host : k_host) + (((long long)u * n + j) * hsp + part);
        v[i] = ld_stream(src);
        dst[i] = (int)(((unsigned)r * CPR + part) * 2u + t);
      }
    }
#pragma unroll
    for (int i = 0; i < INFL; ++i)
      if (dst[i] >= 0) ((dst[i] & 1) ? v_buf : k_buf)[dst[i] >> 1] = v[i];
  }
}

template <int CPR>
__global__ void __launch_bounds__(kLsuMaxThreads)
    gather_lsu_kernel(const uint4* __restrict__ k_host, const uint4* __restrict__ v_host,
                      const int32_t* __restrict__ idx, uint4* __restrict__ k_buf,
                      uint4* __restrict__ v_buf, int n, int k, long long rows, long long hsp) {
  gather_lsu_body<CPR, kInFlight>(k_host, v_host, idx, k_buf, v_buf, n, k, rows, hsp);
}

template <int CPR>
cudaError_t launch_lsu(const Dims& d, const HostKV& h, const int32_t* idx, void* kb, void* vb,
                       cudaStream_t st) {
  static unsigned long long prepared = 0;
  const long long rows = (long long)d.U * d.k;
  if (rows * 2 * CPR * 2 >= (1ll << 31)) return cudaErrorInvalidValue;  // piece index range
  cudaError_t e = prepare_kernel(gather_lsu_kernel<CPR>, &prepared, 0);
  if (e != cudaSuccess) return e;
  const int threads = g_lsu_threads.load();
  const long long work = (rows * 2 * CPR + (long long)threads * kInFlight - 1) /
                         ((long long)threads * kInFlight);
  long long grid = ((long long)sm_count() * g_lsu_grid_pct.load() + 99) / 100;
  if (grid > work) grid = work;
  if (grid < 1) grid = 1;
  gather_lsu_kernel<CPR><<<(unsigned)grid, threads, 0, st>>>(
      static_cast<const uint4*>(h.k), static_cast<const uint4*>(h.v), idx,
      static_cast<uint4*>(kb), static_cast<uint4*>(vb), d.n, d.k, rows,
      (long long)(h.hs / 16));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const Dims& d, const HostKV& h, const int32_t* idx, void* k_buf,
                          void* v_buf, int mode, cudaStream_t st, bool touch) {
  const int rb = d.d * d.elt;
  if (touch && (mode == 0 || mode == 1)) {
    static unsigned int* sinks[64] = {};  // device address of g_touch_sink, per device
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    unsigned int*& sink = sinks[dev & 63];
    if (!sink) {
      e0 = cudaGetSymbolAddress(reinterpret_cast<void**>(&sink), g_touch_sink);
      if (e0 != cudaSuccess) return e0;
    }
    // The rows span U n hs bytes from each base (the two ranges overlap in an
    // interleaved store, which touches its pages twice: harmless).
    const size_t bytes = (size_t)d.U * d.n * h.hs - (h.hs - rb);
    touch_pages_kernel<<<1, 32, 0, st>>>(static_cast<const unsigned char*>(h.k),
                                         static_cast<const unsigned char*>(h.v), bytes,
                                         host_page_bytes(), sink);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (mode == 0) {
    switch (rb) {
      case 128: return launch_tma<128>(d, h, idx, k_buf, v_buf, st);
      case 256: return launch_tma<256>(d, h, idx, k_buf, v_buf, st);
      case 512: return launch_tma<512>(d, h, idx, k_buf, v_buf, st);
    }
  } else if (mode == 1) {
    switch (rb / 16) {
      case 8: return launch_lsu<8>(d, h, idx, k_buf, v_buf, st);
      case 16: return launch_lsu<16>(d, h, idx, k_buf, v_buf, st);
      case 32: return launch_lsu<32>(d, h, idx, k_buf, v_buf, st);
    }
  }
  return cudaErrorInvalidValue;
}

dd_status set_gather_geometry(int grid_pct, int tile_bytes, int stages) {
  if (grid_pct < 1 || grid_pct > 800 || stages < 1 || stages > kMaxStages ||
      tile_bytes < 512 || tile_bytes > kMaxTileBytes || tile_bytes % 512 != 0 ||
      tma_smem(1, tile_bytes, stages) > (size_t)kMaxDynSmem)
    return DD_ERR_INVALID_ARG;
  g_grid_pct.store(grid_pct);
  g_tile_bytes.store(tile_bytes);
  g_stages.store(stages);
  return DD_OK;
}

dd_status set_gather_lsu_geometry(int grid_pct, int threads) {
  if (grid_pct < 1 || grid_pct > 800 || threads < 32 || threads > kLsuMaxThreads ||
      threads % 32 != 0)
    return DD_ERR_INVALID_ARG;
  g_lsu_grid_pct.store(grid_pct);
  g_lsu_threads.store(threads);
  return DD_OK;
}

unsigned int take_gather_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gather_status, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_gather_status, &zero, sizeof zero);
  return v;
}

}  // namespace dd
