// C ABI of libdd.so: argument checks, workspace layout, the three per-layer
// calls and the two-stream layer loop with its double-buffered, layer-scoped
// scratch (DualDecoder paper Sec. 1: layer-aware transfer schedule and
// layer-scoped KV memory manager; summary page: transfer time
// T_transfer = sum_l S_l / B hidden by min max(T_compute, T_transfer), and the
// runtime sparse-KV buffer reduced from O(n d) to O(k d)).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include <cstdio>
#include <initializer_list>
#include <map>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "dd_internal.cuh"

#define DD_VERSION 10000

namespace dd {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

dd_status resolve(const dd_shape* s, Dims* o) {
  if (!s || !o) return DD_ERR_INVALID_ARG;
  if (s->batch < 1 || s->n_q_heads < 1 || s->n_kv_heads < 1 || s->head_dim < 1 ||
      s->ctx_len < 1 || s->top_k < 1 || s->window < 0)
    return DD_ERR_INVALID_ARG;
  if (s->n_q_heads % s->n_kv_heads != 0) return DD_ERR_INVALID_ARG;
  if (s->window >= s->ctx_len) return DD_ERR_INVALID_ARG;
  if (s->top_k > s->ctx_len - s->window) return DD_ERR_INVALID_ARG;
  if (s->dtype != DD_F32 && s->dtype != DD_BF16) return DD_ERR_UNSUPPORTED;
  const int G = s->n_q_heads / s->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return DD_ERR_UNSUPPORTED;
  if (s->ctx_len > (1 << 30)) return DD_ERR_UNSUPPORTED;
  const int chunk =
      score_chunk(s->dtype, s->head_dim, (long long)s->batch * s->n_kv_heads, s->ctx_len);
  if (chunk == 0) return DD_ERR_UNSUPPORTED;
  Dims d;
  d.B = s->batch;
  d.Hq = s->n_q_heads;
  d.Hkv = s->n_kv_heads;
  d.G = G;
  d.d = s->head_dim;
  d.n = s->ctx_len;
  d.k = s->top_k;
  d.W = s->window;
  d.dtype = s->dtype;
  d.elt = s->dtype == DD_BF16 ? 2 : 4;
  const long long U = (long long)d.B * d.Hkv;
  if (U > (1 << 24)) return DD_ERR_UNSUPPORTED;
  d.U = (int)U;
  d.span = d.n - d.W;
  d.ldn = (d.n + 3) & ~3;
  d.chunk = chunk;
  d.nchunks = (d.n + chunk - 1) / chunk;
  if ((long long)d.U * d.nchunks > 0x7FFFFFFFLL) return DD_ERR_UNSUPPORTED;
  d.rows = d.k + d.W;
  d.nsplit = (d.rows + kAttnRowsPerSplit - 1) / kAttnRowsPerSplit;
  if ((long long)d.U * d.k > 0x7FFFFFFFLL) return DD_ERR_UNSUPPORTED;
  *o = d;
  return DD_OK;
}

WsLayout ws_layout(const Dims& d) {
  WsLayout w;
  size_t off = 0;
  w.logits = off;
  off += align256((size_t)d.B * d.Hq * d.ldn * sizeof(float));
  w.part = off;
  off += align256((size_t)d.B * d.Hq * d.nchunks * sizeof(float2));
  w.attn_o = off;
  off += align256((size_t)d.B * d.Hq * d.nsplit * d.d * sizeof(float));
  w.attn_ml = off;
  off += align256((size_t)d.B * d.Hq * d.nsplit * sizeof(float2));
  w.sel_true = off;
  off += align256((size_t)d.U * d.k * sizeof(float));
  w.counters = off;
  off += align256((size_t)d.U * sizeof(int32_t));
  w.attn_counters = off;
  off += align256((size_t)d.U * sizeof(int32_t));
  w.total = off;
  return w;
}

cudaError_t select_rows(const Dims& d, const WsLayout& lay, char* ws, const void* q,
                        const void* k_dev, int32_t* idx, float* sel, float* lse, bool fused,
                        cudaStream_t st, int* launches) {
  float* logits = reinterpret_cast<float*>(ws + lay.logits);
  float2* part = reinterpret_cast<float2*>(ws + lay.part);
  if (fused) {
    *launches += kScoreSelectLaunches;
    return launch_score_select(d, q, k_dev, logits, part,
                               reinterpret_cast<int32_t*>(ws + lay.counters), idx, sel, lse, st);
  }
  *launches += kScoreLaunches + kTopkLaunches;
  cudaError_t e = launch_score(d, q, k_dev, logits, part, st);
  if (e == cudaSuccess) e = launch_topk(d, logits, part, idx, sel, lse, st);
  return e;
}



dd_status resolve_landmarks(const dd_shape* s, int chunk, LandmarkDims* out) {
  Dims f;
  dd_status st = resolve(s, &f);
  if (st != DD_OK) return st;
  if (chunk < 2 || f.span % chunk != 0 || f.k % chunk != 0) return DD_ERR_UNSUPPORTED;
  if (f.d != 64 && f.d != 128) return DD_ERR_UNSUPPORTED;  // fp32 landmark rows <= 512 B
  dd_shape ls = *s;
  ls.ctx_len = f.span / chunk;
  ls.top_k = f.k / chunk;
  ls.window = 0;
  ls.dtype = DD_F32;
  LandmarkDims L;
  st = resolve(&ls, &L.lm);
  if (st != DD_OK) return st;
  L.full = f;
  L.chunk = chunk;
  L.lay = ws_layout(L.lm);
  L.q32 = L.lay.total;
  L.chunks = L.q32 + align256((size_t)f.B * f.Hq * f.d * sizeof(float));
  L.total = L.chunks + align256((size_t)f.U * L.lm.k * sizeof(int32_t));
  *out = L;
  return DD_OK;
}

// Device memory of the current device, or managed memory.
bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  int dev = -1;
  return a.type == cudaMemoryTypeDevice && cudaGetDevice(&dev) == cudaSuccess && a.device == dev;
}

bool lsu_gather_fits(const Dims& d) {
  return (long long)d.U * d.k * d.d * d.elt < (8ll << 30);  // 16-byte piece index range
}

bool all_device(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !is_device_ptr(p)) return false;
  return true;
}

}  // namespace dd

using namespace dd;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

dd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DD_OK : DD_ERR_CUDA; }

}  // namespace

extern "C" {

const char* dd_status_string(int s) {
  switch (s) {
    case DD_OK: return "ok";
    case DD_ERR_INVALID_ARG: return "invalid argument";
    case DD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case DD_ERR_OOM: return "device allocation failed";
    case DD_ERR_CUDA: return "CUDA runtime error";
    case DD_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int dd_version(void) { return DD_VERSION; }

dd_status dd_check_device(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return DD_ERR_CUDA;
  const unsigned int a = take_score_status();
  const unsigned int b = take_gather_status();
  const unsigned int c = take_debug_status();
  return (a | b | c) ? DD_ERR_TIMEOUT : DD_OK;
}

dd_status dd_debug_expire_wait(uint64_t limit_ns, dd_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 100000000ull) return DD_ERR_INVALID_ARG;
  return cuda_status(launch_expire_wait(limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

dd_status dd_set_gather_geometry(int grid_pct, int tile_bytes, int stages) {
  return set_gather_geometry(grid_pct, tile_bytes, stages);
}

dd_status dd_set_gather_lsu_geometry(int grid_pct, int threads) {
  return set_gather_lsu_geometry(grid_pct, threads);
}

int dd_score_tensor_cores(const dd_shape* shape) {
  Dims d;
  const dd_status st = resolve(shape, &d);
  if (st != DD_OK) return -(int)st;
  return score_uses_mma(d.dtype, d.G) ? 1 : 0;
}

dd_status dd_workspace_size(const dd_shape* shape, size_t* bytes) {
  if (!bytes) return DD_ERR_INVALID_ARG;
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  *bytes = ws_layout(d).total;
  return DD_OK;
}

dd_status dd_score_topk(const dd_shape* shape, const void* q_spec, const void* k_dev,
                        int32_t* idx_out, float* sel_score_out, float* lse_out, void* workspace,
                        size_t ws_bytes, dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (!q_spec || !k_dev || !idx_out || !sel_score_out || !workspace) return DD_ERR_INVALID_ARG;
  if (!aligned16(q_spec) || !aligned16(k_dev) || !aligned16(workspace)) return DD_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  if (ws_bytes < w.total) return DD_ERR_INVALID_ARG;
  if (!all_device({q_spec, k_dev, idx_out, sel_score_out, lse_out, workspace}))
    return DD_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int launches = 0;
  return cuda_status(
      select_rows(d, w, ws, q_spec, k_dev, idx_out, sel_score_out, lse_out, false, s, &launches));
}

dd_status dd_gather_h2d(const dd_shape* shape, const void* k_host, const void* v_host,
                        const int32_t* idx, void* k_buf, void* v_buf, int mode,
                        dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (mode != 0 && mode != 1) return DD_ERR_UNSUPPORTED;
  if (mode == 1 && !lsu_gather_fits(d)) return DD_ERR_UNSUPPORTED;
  if (!k_host || !v_host || !idx || !k_buf || !v_buf) return DD_ERR_INVALID_ARG;
  if (!aligned16(k_host) || !aligned16(v_host) || !aligned16(k_buf) || !aligned16(v_buf))
    return DD_ERR_INVALID_ARG;
  const void* kh = host_to_device(k_host);
  const void* vh = host_to_device(v_host);
  if (!kh || !vh) return DD_ERR_INVALID_ARG;
  if (!all_device({idx, k_buf, v_buf})) return DD_ERR_INVALID_ARG;
  const bool touch = in_huge_page_store(k_host) || in_huge_page_store(v_host);
  const HostKV h{kh, vh, (size_t)d.d * d.elt};
  return cuda_status(launch_gather(d, h, idx, k_buf, v_buf, mode,
                                   reinterpret_cast<cudaStream_t>(stream), touch));
}

dd_status dd_gather_h2d_kv(const dd_shape* shape, const void* kv_host, const int32_t* idx,
                           void* k_buf, void* v_buf, int mode, dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (mode != 0 && mode != 1) return DD_ERR_UNSUPPORTED;
  if (mode == 1 && !lsu_gather_fits(d)) return DD_ERR_UNSUPPORTED;
  if (!kv_host || !idx || !k_buf || !v_buf) return DD_ERR_INVALID_ARG;
  if (!aligned16(kv_host) || !aligned16(k_buf) || !aligned16(v_buf)) return DD_ERR_INVALID_ARG;
  const void* kvh = host_to_device(kv_host);
  if (!kvh) return DD_ERR_INVALID_ARG;
  if (!all_device({idx, k_buf, v_buf})) return DD_ERR_INVALID_ARG;
  const size_t rb = (size_t)d.d * d.elt;
  const HostKV h{kvh, static_cast<const char*>(kvh) + rb, 2 * rb};
  return cuda_status(launch_gather(d, h, idx, k_buf, v_buf, mode,
                                   reinterpret_cast<cudaStream_t>(stream),
                                   in_huge_page_store(kv_host)));
}

dd_status dd_sparse_decode_attn(const dd_shape* shape, const void* q, const void* k_buf,
                                const void* v_buf, const void* k_dev, const void* v_win,
                                float* out, void* workspace, size_t ws_bytes,
                                dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (!q || !k_buf || !v_buf || !k_dev || !out || !workspace) return DD_ERR_INVALID_ARG;
  if (d.W > 0 && !v_win) return DD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(k_dev) ||
      !aligned16(out) || !aligned16(workspace) || (v_win && !aligned16(v_win)))
    return DD_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  if (ws_bytes < w.total) return DD_ERR_INVALID_ARG;
  if (!all_device({q, k_buf, v_buf, k_dev, v_win, out, workspace})) return DD_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  return cuda_status(launch_attn(d, q, k_buf, v_buf, window_in_cache(k_dev, d), v_win, out,
                                 reinterpret_cast<float*>(ws + w.attn_o),
                                 reinterpret_cast<float2*>(ws + w.attn_ml),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// Miss correction against a host store described by `h` (rows already
// translated to device-accessible addresses; h.k == NULL if the store was not
// page-locked host memory).
dd_status correct_misses(const dd_shape* shape, const void* q, const void* k_dev,
                         const int32_t* idx_spec, const void* k_buf_spec, const void* v_buf_spec,
                         const HostKV& h, int32_t* idx_true_out, void* k_buf_out,
                         void* v_buf_out, int32_t* miss_out, float* mass_out, void* workspace,
                         size_t ws_bytes, dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (d.k > kMaxCorrectK) return DD_ERR_UNSUPPORTED;
  if (!q || !k_dev || !idx_spec || !k_buf_spec || !v_buf_spec || !idx_true_out || !k_buf_out ||
      !v_buf_out || !workspace)
    return DD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_dev) || !aligned16(k_buf_spec) || !aligned16(v_buf_spec) ||
      !aligned16(k_buf_out) || !aligned16(v_buf_out) || !aligned16(workspace))
    return DD_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  if (ws_bytes < w.total) return DD_ERR_INVALID_ARG;
  if (!h.k || !h.v) return DD_ERR_INVALID_ARG;
  if (!all_device({q, k_dev, idx_spec, k_buf_spec, v_buf_spec, idx_true_out, k_buf_out, v_buf_out,
                   miss_out, mass_out, workspace}))
    return DD_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* sel_true = reinterpret_cast<float*>(ws + w.sel_true);
  int launches = 0;
  st = cuda_status(
      select_rows(d, w, ws, q, k_dev, idx_true_out, sel_true, nullptr, false, s, &launches));
  if (st != DD_OK) return st;
  return cuda_status(launch_fixup(d, idx_spec, idx_true_out, sel_true, k_buf_spec, v_buf_spec, h,
                                  k_buf_out, v_buf_out, miss_out, mass_out, s));
}
}  // namespace

extern "C" {

dd_status dd_correct_misses(const dd_shape* shape, const void* q, const void* k_dev,
                            const int32_t* idx_spec, const void* k_buf_spec,
                            const void* v_buf_spec, const void* k_host, const void* v_host,
                            int32_t* idx_true_out, void* k_buf_out, void* v_buf_out,
                            int32_t* miss_out, float* mass_out, void* workspace, size_t ws_bytes,
                            dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (d.k > kMaxCorrectK) return DD_ERR_UNSUPPORTED;
  if (!k_host || !v_host || !aligned16(k_host) || !aligned16(v_host)) return DD_ERR_INVALID_ARG;
  const HostKV h{host_to_device(k_host), host_to_device(v_host), (size_t)d.d * d.elt};
  return correct_misses(shape, q, k_dev, idx_spec, k_buf_spec, v_buf_spec, h, idx_true_out,
                        k_buf_out, v_buf_out, miss_out, mass_out, workspace, ws_bytes, stream);
}

dd_status dd_correct_misses_kv(const dd_shape* shape, const void* q, const void* k_dev,
                               const int32_t* idx_spec, const void* k_buf_spec,
                               const void* v_buf_spec, const void* kv_host,
                               int32_t* idx_true_out, void* k_buf_out, void* v_buf_out,
                               int32_t* miss_out, float* mass_out, void* workspace,
                               size_t ws_bytes, dd_stream_t stream) {
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  if (d.k > kMaxCorrectK) return DD_ERR_UNSUPPORTED;
  if (!kv_host || !aligned16(kv_host)) return DD_ERR_INVALID_ARG;
  const size_t rb = (size_t)d.d * d.elt;
  const void* kvh = host_to_device(kv_host);
  const HostKV h{kvh, kvh ? static_cast<const char*>(kvh) + rb : nullptr, 2 * rb};
  return correct_misses(shape, q, k_dev, idx_spec, k_buf_spec, v_buf_spec, h, idx_true_out,
                        k_buf_out, v_buf_out, miss_out, mass_out, workspace, ws_bytes, stream);
}

dd_status dd_landmarks_size(const dd_shape* shape, int chunk, size_t* bytes) {
  if (!bytes) return DD_ERR_INVALID_ARG;
  LandmarkDims L;
  dd_status st = resolve_landmarks(shape, chunk, &L);
  if (st != DD_OK) return st;
  *bytes = (size_t)L.full.U * L.lm.n * L.full.d * sizeof(float);
  return DD_OK;
}

dd_status dd_landmarks_workspace_size(const dd_shape* shape, int chunk, size_t* bytes) {
  if (!bytes) return DD_ERR_INVALID_ARG;
  LandmarkDims L;
  dd_status st = resolve_landmarks(shape, chunk, &L);
  if (st != DD_OK) return st;
  *bytes = L.total;
  return DD_OK;
}

dd_status dd_build_landmarks(const dd_shape* shape, int chunk, const void* k_dev,
                             float* landmarks_out, dd_stream_t stream) {
  LandmarkDims L;
  dd_status st = resolve_landmarks(shape, chunk, &L);
  if (st != DD_OK) return st;
  if (!k_dev || !landmarks_out) return DD_ERR_INVALID_ARG;
  if (!aligned16(k_dev) || !aligned16(landmarks_out)) return DD_ERR_INVALID_ARG;
  if (!all_device({k_dev, landmarks_out})) return DD_ERR_INVALID_ARG;
  return cuda_status(
      launch_landmarks(L.full, chunk, k_dev, landmarks_out, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// Landmark selection into `rows` (the k expanded rows) and `sel` (chunk scores).
// The fused selection's counters in `ws` must be zero (they are after it).
cudaError_t landmark_select(const LandmarkDims& L, const void* q, const void* landmarks,
                            int32_t* rows, float* sel, float* lse, char* ws, bool fused,
                            cudaStream_t st, int* launches) {
  const Dims& f = L.full;
  if (!fused) {
    // Scoring reads the bf16 query itself; the top-k writes each selected
    // chunk's rows.
    float* logits = reinterpret_cast<float*>(ws + L.lay.logits);
    float2* part = reinterpret_cast<float2*>(ws + L.lay.part);
    cudaError_t e = f.dtype == DD_BF16
                        ? launch_score_bf16_query(L.lm, q, landmarks, logits, part, st)
                        : launch_score(L.lm, q, landmarks, logits, part, st);
    if (e == cudaSuccess) e = launch_topk(L.lm, logits, part, rows, sel, lse, st, L.chunk);
    *launches += kScoreLaunches + kTopkLaunches;
    return e;
  }
  const float* q32 = static_cast<const float*>(q);
  if (f.dtype == DD_BF16) {
    float* tmp = reinterpret_cast<float*>(ws + L.q32);
    cudaError_t e = launch_to_f32(q, tmp, f.B * f.Hq * f.d, st);
    if (e != cudaSuccess) return e;
    q32 = tmp;
    ++*launches;
  }
  int32_t* chunks = reinterpret_cast<int32_t*>(ws + L.chunks);
  cudaError_t e = select_rows(L.lm, L.lay, ws, q32, landmarks, chunks, sel, lse, fused, st,
                              launches);
  if (e == cudaSuccess) e = launch_expand(chunks, rows, f.U, L.lm.k, L.chunk, st);
  ++*launches;
  return e;
}
}  // namespace

dd_status dd_score_topk_landmarks(const dd_shape* shape, int chunk, const void* q_spec,
                                  const float* landmarks, int32_t* idx_out, float* chunk_score_out,
                                  float* lse_out, void* workspace, size_t ws_bytes,
                                  dd_stream_t stream) {
  LandmarkDims L;
  dd_status st = resolve_landmarks(shape, chunk, &L);
  if (st != DD_OK) return st;
  if (!q_spec || !landmarks || !idx_out || !chunk_score_out || !workspace)
    return DD_ERR_INVALID_ARG;
  if (!aligned16(q_spec) || !aligned16(landmarks) || !aligned16(workspace))
    return DD_ERR_INVALID_ARG;
  if (ws_bytes < L.total) return DD_ERR_INVALID_ARG;
  if (!all_device({q_spec, landmarks, idx_out, chunk_score_out, lse_out, workspace}))
    return DD_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int launches = 0;
  return cuda_status(landmark_select(L, q_spec, landmarks, idx_out, chunk_score_out, lse_out, ws,
                                     false, s, &launches));
}

}  // extern "C"

// ------------------------------------------------------------------ context

constexpr int kMaxTimingDepth = 4096;

enum Phase { PH_SCORE0, PH_SCORE1, PH_TOPK1, PH_GATHER0, PH_GATHER1, PH_ATTN0, PH_ATTN1, PH_N };

// The events of one timed step: PH_N per layer, plus the step's first and last.
struct TimingSet {
  std::vector<cudaEvent_t> tev;
  cudaEvent_t t_begin = nullptr, t_end = nullptr;
  int layers = 0;
  int launches = 0;
  bool light = false;  // DD_STEP_TIMING_LIGHT: only the scoring events
  void release() {
    for (cudaEvent_t e : tev) cudaEventDestroy(e);
    tev.clear();
    if (t_begin) cudaEventDestroy(t_begin);
    if (t_end) cudaEventDestroy(t_end);
    t_begin = t_end = nullptr;
  }
};

struct dd_ctx {
  dd_shape shape;
  Dims dims;
  WsLayout ws_lay;
  int device;
  void* kbuf[2];
  void* vbuf[2];
  int32_t* idx[2];
  float* sel[2];
  float* lse;
  void* ws;
  size_t device_bytes;
  cudaEvent_t ev_idx[2], ev_ready[2], ev_free[2], ev_join;
  // Timing: per layer PH_N events, plus the step's first and last.
  // A ring of t_depth event sets: timed step i records into set i % t_depth,
  // so the last t_depth timed steps can be read without a host wait between
  // steps.  t_last is the set of the last timed step, t_count how many timed
  // steps the ring holds.
  std::vector<TimingSet> tsets;
  int t_depth;
  int t_last;
  int t_count;
  // Miss correction (DD_STEP_CORRECT_MISSES): the real query's indices and
  // rows, and per-layer statistics, grown to the largest layer count used.
  int32_t* idx_true;
  void* kb_true;
  void* vb_true;
  int32_t* miss;  // [layers][U]
  float* mass;    // [layers][U][2]: predicted, total
  int corr_layers;
  int last_corr_layers;
  cudaEvent_t ev_done;
  // Landmark selection (DD_STEP_LANDMARKS), set by dd_ctx_set_landmark_chunk.
  int lm_chunk;
  LandmarkDims lm;
  void* lm_ws;  // its own workspace: under DD_STEP_PIPELINE the selection of
                // layer l+1 runs beside the attention of layer l
  // A captured decode step (dd_ctx_capture_step), replayed by dd_ctx_replay_step.
  cudaGraph_t graph;
  cudaGraphExec_t graph_exec;
  int graph_launches;
};

namespace {

void ctx_free(dd_ctx* c) {
  if (!c) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(c->device);
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  for (int i = 0; i < 2; ++i) {
    cudaFree(c->kbuf[i]);
    cudaFree(c->vbuf[i]);
    cudaFree(c->idx[i]);
    cudaFree(c->sel[i]);
    if (c->ev_idx[i]) cudaEventDestroy(c->ev_idx[i]);
    if (c->ev_ready[i]) cudaEventDestroy(c->ev_ready[i]);
    if (c->ev_free[i]) cudaEventDestroy(c->ev_free[i]);
  }
  cudaFree(c->lse);
  cudaFree(c->ws);
  cudaFree(c->idx_true);
  cudaFree(c->kb_true);
  cudaFree(c->vb_true);
  cudaFree(c->miss);
  cudaFree(c->mass);
  cudaFree(c->lm_ws);
  if (c->ev_done) cudaEventDestroy(c->ev_done);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  for (TimingSet& t : c->tsets) t.release();
  if (prev >= 0) cudaSetDevice(prev);
  delete c;
}

dd_status ensure_correction_buffers(dd_ctx* c, int n_layers) {
  const Dims& d = c->dims;
  if (!c->idx_true) {
    const size_t rows_bytes = (size_t)d.U * d.k * d.d * d.elt;
    if (cudaMalloc((void**)&c->idx_true, (size_t)d.U * d.k * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&c->kb_true, rows_bytes) != cudaSuccess ||
        cudaMalloc(&c->vb_true, rows_bytes) != cudaSuccess) {
      cudaGetLastError();
      return DD_ERR_OOM;
    }
    c->device_bytes += (size_t)d.U * d.k * sizeof(int32_t) + 2 * rows_bytes;
  }
  if (n_layers > c->corr_layers) {
    cudaFree(c->miss);
    cudaFree(c->mass);
    c->miss = nullptr;
    c->mass = nullptr;
    if (cudaMalloc((void**)&c->miss, (size_t)n_layers * d.U * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc((void**)&c->mass, (size_t)n_layers * d.U * 2 * sizeof(float)) != cudaSuccess) {
      cudaGetLastError();
      c->corr_layers = 0;
      return DD_ERR_OOM;
    }
    c->corr_layers = n_layers;
  }
  return DD_OK;
}

dd_status ensure_timing_events(TimingSet& t, int n_layers) {
  const size_t need = (size_t)n_layers * PH_N;
  while (t.tev.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return DD_ERR_CUDA;
    t.tev.push_back(e);
  }
  if (!t.t_begin && cudaEventCreate(&t.t_begin) != cudaSuccess) return DD_ERR_CUDA;
  if (!t.t_end && cudaEventCreate(&t.t_end) != cudaSuccess) return DD_ERR_CUDA;
  return DD_OK;
}

// The timing set of the timed step `back` steps before the last one.
TimingSet* timing_set(dd_ctx* c, int back) {
  if (back < 0 || back >= c->t_count) return nullptr;
  TimingSet* t = &c->tsets[(size_t)((c->t_last - back + c->t_depth) % c->t_depth)];
  if (cudaEventSynchronize(t->t_end) != cudaSuccess) return nullptr;
  return t;
}

}  // namespace

extern "C" {

dd_status dd_ctx_create(const dd_shape* shape, dd_ctx** out) {
  if (!out) return DD_ERR_INVALID_ARG;
  *out = nullptr;
  Dims d;
  dd_status st = resolve(shape, &d);
  if (st != DD_OK) return st;
  dd_ctx* c = new (std::nothrow) dd_ctx();
  if (!c) return DD_ERR_OOM;
  c->shape = *shape;
  c->dims = d;
  c->tsets.resize(1);
  c->t_depth = 1;
  c->t_last = -1;
  c->t_count = 0;
  c->ws_lay = ws_layout(d);
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    delete c;
    return DD_ERR_CUDA;
  }
  const size_t rows_bytes = (size_t)d.U * d.k * d.d * d.elt;
  const size_t idx_bytes = (size_t)d.U * d.k * sizeof(int32_t);
  const size_t sel_bytes = (size_t)d.U * d.k * sizeof(float);
  bool ok = true;
  for (int i = 0; i < 2 && ok; ++i) {
    ok = cudaMalloc(&c->kbuf[i], rows_bytes) == cudaSuccess &&
         cudaMalloc(&c->vbuf[i], rows_bytes) == cudaSuccess &&
         cudaMalloc((void**)&c->idx[i], idx_bytes) == cudaSuccess &&
         cudaMalloc((void**)&c->sel[i], sel_bytes) == cudaSuccess;
  }
  ok = ok && cudaMalloc((void**)&c->lse, (size_t)d.B * d.Hq * sizeof(float)) == cudaSuccess;
  ok = ok && cudaMalloc(&c->ws, c->ws_lay.total) == cudaSuccess;
  // The fused selection's and the attention merge's counters start at zero
  // (each launch leaves them so).
  ok = ok &&
       cudaMemset(static_cast<char*>(c->ws) + c->ws_lay.counters, 0,
                  (size_t)d.U * sizeof(int32_t)) == cudaSuccess &&
       cudaMemset(static_cast<char*>(c->ws) + c->ws_lay.attn_counters, 0,
                  (size_t)d.U * sizeof(int32_t)) == cudaSuccess &&
       cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    ctx_free(c);
    return DD_ERR_OOM;
  }
  c->device_bytes = 2 * (2 * rows_bytes + idx_bytes + sel_bytes) +
                    (size_t)d.B * d.Hq * sizeof(float) + c->ws_lay.total;
  for (int i = 0; i < 2 && ok; ++i)
    ok = cudaEventCreateWithFlags(&c->ev_idx[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&c->ev_ready[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&c->ev_free[i], cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    ctx_free(c);
    return DD_ERR_CUDA;
  }
  *out = c;
  return DD_OK;
}

void dd_ctx_destroy(dd_ctx* ctx) { ctx_free(ctx); }

size_t dd_ctx_device_bytes(const dd_ctx* ctx) { return ctx ? ctx->device_bytes : 0; }

dd_status dd_ctx_set_landmark_chunk(dd_ctx* c, int chunk) {
  if (!c) return DD_ERR_INVALID_ARG;
  LandmarkDims L;
  dd_status st = resolve_landmarks(&c->shape, chunk, &L);
  if (st != DD_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) return DD_ERR_INVALID_ARG;
  const size_t have = c->lm_chunk ? c->lm.total : 0;
  if (L.total > have) {
    cudaDeviceSynchronize();  // a step may still use the old buffer
    cudaFree(c->lm_ws);
    c->device_bytes -= have;
    c->lm_ws = nullptr;
    c->lm_chunk = 0;
    if (cudaMalloc(&c->lm_ws, L.total) != cudaSuccess) {
      c->lm_ws = nullptr;
      cudaGetLastError();
      return DD_ERR_OOM;
    }
    c->device_bytes += L.total;
  } else {
    L.total = have;  // keep the larger buffer's size on record
    cudaDeviceSynchronize();  // a step may still use the buffer in its old layout
  }
  // The fused selection's counters of this layout start at zero (in a reused
  // buffer that memory held something else).
  if (cudaMemset(static_cast<char*>(c->lm_ws) + L.lay.counters, 0,
                 (size_t)L.lm.U * sizeof(int32_t)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    c->lm_chunk = 0;
    return DD_ERR_CUDA;
  }
  c->lm = L;
  c->lm_chunk = chunk;
  return DD_OK;
}

dd_status dd_decode_step(dd_ctx* c, const dd_layer_io* layers, int n_layers,
                         dd_stream_t compute, dd_stream_t copy, int flags) {
  if (!c || !layers || n_layers < 1) return DD_ERR_INVALID_ARG;
  int cur_dev = -1;
  if (cudaGetDevice(&cur_dev) != cudaSuccess || cur_dev != c->device) return DD_ERR_INVALID_ARG;
  const Dims& d = c->dims;
  // Synchronous checks of every layer before anything is enqueued.
  std::vector<HostKV> hkv(n_layers);
  std::vector<char> touch(n_layers);
  const size_t rb = (size_t)d.d * d.elt;
  // Without DD_STEP_LANDMARKS the key cache is scored, so k_dev is required;
  // with it, k_dev is needed only for the window's keys, if k_win is NULL.
  const bool lm_flag = (flags & DD_STEP_LANDMARKS) != 0;
  for (int l = 0; l < n_layers; ++l) {
    const dd_layer_io& io = layers[l];
    if (!io.q_spec || !io.q || !io.out) return DD_ERR_INVALID_ARG;
    // The host store: separate K and V stores, or one interleaved store.
    if (io.kv_host ? (io.k_host || io.v_host) : (!io.k_host || !io.v_host))
      return DD_ERR_INVALID_ARG;
    if (!io.k_dev && !(lm_flag && (io.k_win || d.W == 0))) return DD_ERR_INVALID_ARG;
    if (d.W > 0 && !io.v_win) return DD_ERR_INVALID_ARG;
    if (!aligned16(io.q_spec) || !aligned16(io.q) || !aligned16(io.k_dev) ||
        !aligned16(io.k_host) || !aligned16(io.v_host) || !aligned16(io.kv_host) ||
        !aligned16(io.out) ||
        !aligned16(io.v_win) || !aligned16(io.k_win))
      return DD_ERR_INVALID_ARG;
    if (io.kv_host) {
      const void* kvh = host_to_device(io.kv_host);
      if (!kvh) return DD_ERR_INVALID_ARG;
      hkv[l] = HostKV{kvh, static_cast<const char*>(kvh) + rb, 2 * rb};
      touch[l] = in_huge_page_store(io.kv_host);
    } else {
      hkv[l] = HostKV{host_to_device(io.k_host), host_to_device(io.v_host), rb};
      if (!hkv[l].k || !hkv[l].v) return DD_ERR_INVALID_ARG;
      touch[l] = in_huge_page_store(io.k_host) || in_huge_page_store(io.v_host);
    }
    if (!all_device({io.q_spec, io.q, io.k_dev, io.v_win, io.k_win, io.out}))
      return DD_ERR_INVALID_ARG;
  }
  const bool light = (flags & DD_STEP_TIMING_LIGHT) != 0;
  const bool timing = light || (flags & DD_STEP_TIMING) != 0;
  const bool phases = timing && !light;  // the events of every phase
  const int gather_mode = (flags & DD_STEP_GATHER_LSU) ? 1 : 0;
  if (gather_mode == 1 && !lsu_gather_fits(d)) return DD_ERR_UNSUPPORTED;
  const bool correct = (flags & DD_STEP_CORRECT_MISSES) != 0;
  const bool use_lm = (flags & DD_STEP_LANDMARKS) != 0;
  const bool fused = (flags & DD_STEP_FUSED_TOPK) != 0;
  if ((flags & DD_STEP_PIPELINE) &&
      (flags & (DD_STEP_LATE_GATHER | DD_STEP_GATHER_BESIDE_ATTN)))
    return DD_ERR_UNSUPPORTED;  // schedules that exclude each other
  const bool delay_copy = (flags & DD_STEP_DEBUG_DELAY_COPY) != 0;
  const bool delay_compute = (flags & DD_STEP_DEBUG_DELAY_COMPUTE) != 0;
  constexpr uint64_t kDebugDelayNs = 50000;  // 50 us before each gather / attention
  if (use_lm) {
    if (c->lm_chunk == 0 || correct) return DD_ERR_UNSUPPORTED;
    for (int l = 0; l < n_layers; ++l) {
      if (!layers[l].landmarks || !aligned16(layers[l].landmarks)) return DD_ERR_INVALID_ARG;
      if (!all_device({layers[l].landmarks})) return DD_ERR_INVALID_ARG;
    }
  }
  if (correct) {
    if (d.k > kMaxCorrectK) return DD_ERR_UNSUPPORTED;
    if ((flags & DD_STEP_PIPELINE) && copy && copy != compute) return DD_ERR_UNSUPPORTED;
    dd_status st = ensure_correction_buffers(c, n_layers);
    if (st != DD_OK) return st;
  }
  TimingSet* ts = nullptr;
  int t_slot = 0;
  if (timing) {
    t_slot = (c->t_last + 1) % c->t_depth;
    ts = &c->tsets[(size_t)t_slot];
    dd_status st = ensure_timing_events(*ts, n_layers);
    if (st != DD_OK) return st;
  }
  cudaStream_t C = reinterpret_cast<cudaStream_t>(compute);
  cudaStream_t X = copy ? reinterpret_cast<cudaStream_t>(copy) : C;
  const bool serial = (X == C);
  char* ws = static_cast<char*>(c->ws);
  float* logits = reinterpret_cast<float*>(ws + c->ws_lay.logits);
  float2* part = reinterpret_cast<float2*>(ws + c->ws_lay.part);
  float* attn_o = reinterpret_cast<float*>(ws + c->ws_lay.attn_o);
  float2* attn_ml = reinterpret_cast<float2*>(ws + c->ws_lay.attn_ml);
  auto T = [&](int l, int ph) { return ts->tev[(size_t)l * PH_N + ph]; };
  int launches = 0;
#define DD_TRY(x)                                   \
  do {                                              \
    cudaError_t e_ = (x);                           \
    if (e_ != cudaSuccess) return DD_ERR_CUDA;      \
  } while (0)

  // Steps 1-2 of layer l into index slot l % 2 (on the compute stream).
  auto score_topk = [&](int l) -> cudaError_t {
    const int s = l & 1;
    if (timing) cudaEventRecord(T(l, PH_SCORE0), C);
    if (use_lm) {
      // Landmark selection: phase "score" covers it all, "top-k" is empty.
      cudaError_t e = landmark_select(c->lm, layers[l].q_spec, layers[l].landmarks, c->idx[s],
                                      c->sel[s], c->lse, static_cast<char*>(c->lm_ws), fused, C,
                                      &launches);
      if (e != cudaSuccess) return e;
      if (timing) cudaEventRecord(T(l, PH_SCORE1), C);
      if (phases) cudaEventRecord(T(l, PH_TOPK1), C);
      return cudaEventRecord(c->ev_idx[s], C);
    }
    if (fused) {
      // DD_STEP_FUSED_TOPK: one kernel, phase "score" covers the selection.
      cudaError_t e = select_rows(d, c->ws_lay, ws, layers[l].q_spec, layers[l].k_dev, c->idx[s],
                                  c->sel[s], c->lse, true, C, &launches);
      if (e != cudaSuccess) return e;
      if (timing) cudaEventRecord(T(l, PH_SCORE1), C);
      if (phases) cudaEventRecord(T(l, PH_TOPK1), C);
      return cudaEventRecord(c->ev_idx[s], C);
    }
    cudaError_t e = launch_score(d, layers[l].q_spec, layers[l].k_dev, logits, part, C);
    if (e != cudaSuccess) return e;
    if (timing) cudaEventRecord(T(l, PH_SCORE1), C);
    e = launch_topk(d, logits, part, c->idx[s], c->sel[s], c->lse, C);
    if (e != cudaSuccess) return e;
    if (phases) cudaEventRecord(T(l, PH_TOPK1), C);
    launches += kScoreLaunches + kTopkLaunches;
    return cudaEventRecord(c->ev_idx[s], C);
  };
  // Step 3 of layer l into scratch slot l % 2 (on the copy stream).
  auto gather = [&](int l) -> cudaError_t {
    const int s = l & 1;
    cudaError_t e;
    if (!serial) {
      e = cudaStreamWaitEvent(X, c->ev_idx[s], 0);
      if (e != cudaSuccess) return e;
      // The slot's last reader is the attention of layer l - 2 of this step.
      // For l < 2 it belongs to an earlier step, which the copy stream is
      // already ordered after (it waited for all earlier compute work at the
      // start of this step); a wait on that event could not be captured.
      if (l >= 2) {
        e = cudaStreamWaitEvent(X, c->ev_free[s], 0);
        if (e != cudaSuccess) return e;
      }
    }
    if (delay_copy) {
      e = launch_delay(kDebugDelayNs, X);
      if (e != cudaSuccess) return e;
    }
    if (phases) cudaEventRecord(T(l, PH_GATHER0), X);
    e = launch_gather(d, hkv[l], c->idx[s], c->kbuf[s], c->vbuf[s], gather_mode, X, touch[l]);
    if (e != cudaSuccess) return e;
    if (phases) cudaEventRecord(T(l, PH_GATHER1), X);
    launches += kGatherLaunches - (touch[l] ? 0 : 1);
    return cudaEventRecord(c->ev_ready[s], X);
  };
  // Step 4 of layer l from scratch slot l % 2 (on the compute stream).
  // In the pipeline schedule the attention runs on the copy stream, right
  // after the gather of the same layer; otherwise on the compute stream.
  const bool pipeline = !serial && (flags & DD_STEP_PIPELINE) != 0;
  cudaStream_t A = pipeline ? X : C;
  auto attend = [&](int l) -> cudaError_t {
    const int s = l & 1;
    cudaError_t e;
    if (!serial && !pipeline) {
      e = cudaStreamWaitEvent(C, c->ev_ready[s], 0);
      if (e != cudaSuccess) return e;
    }
    if (delay_compute) {
      e = launch_delay(kDebugDelayNs, A);
      if (e != cudaSuccess) return e;
    }
    if (phases) cudaEventRecord(T(l, PH_ATTN0), A);
    const void* kb = c->kbuf[s];
    const void* vb = c->vbuf[s];
    if (correct) {
      // The real query's own top-k; rows the prediction missed come from host.
      float* sel_true = reinterpret_cast<float*>(ws + c->ws_lay.sel_true);
      e = select_rows(d, c->ws_lay, ws, layers[l].q, layers[l].k_dev, c->idx_true, sel_true,
                      nullptr, fused, A, &launches);
      if (e == cudaSuccess)
        e = launch_fixup(d, c->idx[s], c->idx_true, sel_true, c->kbuf[s], c->vbuf[s], hkv[l],
                         c->kb_true, c->vb_true, c->miss + (size_t)l * d.U,
                         c->mass + (size_t)l * d.U * 2, A);
      if (e != cudaSuccess) return e;
      launches += kFixupLaunches;
      kb = c->kb_true;
      vb = c->vb_true;
    }
    const WindowK kw = layers[l].k_win ? window_buffer(layers[l].k_win, d)
                                       : window_in_cache(layers[l].k_dev, d);
    e = launch_attn(d, layers[l].q, kb, vb, kw, layers[l].v_win, layers[l].out, attn_o, attn_ml,
                    A, reinterpret_cast<int32_t*>(ws + c->ws_lay.attn_counters));
    if (e != cudaSuccess) return e;
    if (phases) cudaEventRecord(T(l, PH_ATTN1), A);
    launches += kAttnLaunches - 1;  // the merge runs inside the partial kernel
    return cudaEventRecord(c->ev_free[s], A);
  };

  if (timing) DD_TRY(cudaEventRecord(ts->t_begin, C));
  if (serial) {
    for (int l = 0; l < n_layers; ++l) {
      DD_TRY(score_topk(l));
      DD_TRY(gather(l));
      DD_TRY(attend(l));
    }
  } else if (pipeline) {
    // Two-stage pipeline: compute scores and selects layer after layer; the
    // copy stream gathers and attends each layer as soon as its indices are
    // ready.  Before topk(l) reuses index slot l % 2 (and gather(l) the
    // scratch slot), compute waits for attention(l - 2), the last reader.
    DD_TRY(cudaEventRecord(c->ev_join, C));
    DD_TRY(cudaStreamWaitEvent(X, c->ev_join, 0));
    for (int l = 0; l < n_layers; ++l) {
      if (l >= 2) DD_TRY(cudaStreamWaitEvent(C, c->ev_free[l & 1], 0));
      DD_TRY(score_topk(l));
      DD_TRY(gather(l));
      DD_TRY(attend(l));
    }
    DD_TRY(cudaEventRecord(c->ev_join, X));
    DD_TRY(cudaStreamWaitEvent(C, c->ev_join, 0));
  } else {
    // The copy stream starts after everything already queued on compute
    // (the previous step may still be reading a scratch slot).
    DD_TRY(cudaEventRecord(c->ev_join, C));
    DD_TRY(cudaStreamWaitEvent(X, c->ev_join, 0));
    DD_TRY(score_topk(0));
    DD_TRY(gather(0));
    const bool late = (flags & DD_STEP_LATE_GATHER) != 0;
    const bool guarded = (flags & DD_STEP_GATHER_BESIDE_ATTN) != 0;
    for (int l = 0; l < n_layers; ++l) {
      // Guarded: the next scoring starts only once layer l's gather is done,
      // so a gather runs beside the previous layer's attention, never beside
      // a scoring kernel (the two slow each other down through the memory
      // system's address translation).
      if (guarded) DD_TRY(cudaStreamWaitEvent(C, c->ev_ready[l & 1], 0));
      if (l + 1 < n_layers) DD_TRY(score_topk(l + 1));
      if (l + 1 < n_layers && !late) DD_TRY(gather(l + 1));
      DD_TRY(attend(l));
      if (l + 1 < n_layers && late) {
        // Late gather: layer l+1's rows move only after layer l's attention,
        // so the gather overlaps the scoring of layer l+2, not the attention.
        DD_TRY(cudaStreamWaitEvent(X, c->ev_free[l & 1], 0));
        DD_TRY(gather(l + 1));
      }
    }
    // Join: compute waits for the copy stream's last record.
    DD_TRY(cudaEventRecord(c->ev_join, X));
    DD_TRY(cudaStreamWaitEvent(C, c->ev_join, 0));
  }
  DD_TRY(cudaEventRecord(c->ev_done, C));
  if (correct) c->last_corr_layers = n_layers;
  if (timing) {
    DD_TRY(cudaEventRecord(ts->t_end, C));
    ts->layers = n_layers;
    ts->launches = launches;
    ts->light = light;
    c->t_last = t_slot;
    c->t_count = std::min(c->t_count + 1, c->t_depth);
  }
#undef DD_TRY
  return DD_OK;
}

dd_status dd_ctx_capture_step(dd_ctx* c, const dd_layer_io* layers, int n_layers,
                              dd_stream_t compute, dd_stream_t copy, int flags) {
  if (!c || !layers || n_layers < 1 || !compute) return DD_ERR_INVALID_ARG;
  if (flags & (DD_STEP_TIMING | DD_STEP_TIMING_LIGHT)) return DD_ERR_UNSUPPORTED;
  int cur_dev = -1;
  if (cudaGetDevice(&cur_dev) != cudaSuccess || cur_dev != c->device) return DD_ERR_INVALID_ARG;
  cudaStream_t C = reinterpret_cast<cudaStream_t>(compute);
  // Per-layer buffers that a step allocates on first use must exist before
  // capture (allocation is not captured): run the checks and the lazy
  // allocations outside it, through a step on the caller's stream that is
  // synchronised before capturing.
  dd_status st = dd_decode_step(c, layers, n_layers, compute, copy, flags);
  if (st != DD_OK) return st;
  if (cudaStreamSynchronize(C) != cudaSuccess) return DD_ERR_CUDA;
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  c->graph_exec = nullptr;
  c->graph = nullptr;
  c->graph_launches = 0;
  if (cudaStreamBeginCapture(C, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return DD_ERR_CUDA;
  st = dd_decode_step(c, layers, n_layers, compute, copy, flags);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(C, &g);
  if (st != DD_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return st != DD_OK ? st : DD_ERR_CUDA;
  }
  cudaGraphExec_t x = nullptr;
  if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return DD_ERR_CUDA;
  }
  size_t n_nodes = 0;
  cudaGraphGetNodes(g, nullptr, &n_nodes);
  c->graph = g;
  c->graph_exec = x;
  c->graph_launches = (int)n_nodes;
  return DD_OK;
}

dd_status dd_ctx_replay_step(dd_ctx* c, dd_stream_t stream) {
  if (!c || !c->graph_exec) return DD_ERR_INVALID_ARG;
  int cur_dev = -1;
  if (cudaGetDevice(&cur_dev) != cudaSuccess || cur_dev != c->device) return DD_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(c->graph_exec, reinterpret_cast<cudaStream_t>(stream)));
}

dd_status dd_ctx_step_timings(dd_ctx* c, int back, dd_phase_times* out) {
  if (!c || !out) return DD_ERR_INVALID_ARG;
  TimingSet* t = timing_set(c, back);
  if (!t) return DD_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, t->t_begin, t->t_end) != cudaSuccess) return DD_ERR_CUDA;
  out->step_ms = ms;
  for (int l = 0; l < t->layers; ++l) {
    const cudaEvent_t* e = &t->tev[(size_t)l * PH_N];
    float a = 0.f;
    if (cudaEventElapsedTime(&a, e[PH_SCORE0], e[PH_SCORE1]) != cudaSuccess) return DD_ERR_CUDA;
    out->score_ms += a;
    if (t->light) continue;
    if (cudaEventElapsedTime(&a, e[PH_SCORE1], e[PH_TOPK1]) != cudaSuccess) return DD_ERR_CUDA;
    out->topk_ms += a;
    if (cudaEventElapsedTime(&a, e[PH_GATHER0], e[PH_GATHER1]) != cudaSuccess) return DD_ERR_CUDA;
    out->gather_ms += a;
    if (cudaEventElapsedTime(&a, e[PH_ATTN0], e[PH_ATTN1]) != cudaSuccess) return DD_ERR_CUDA;
    out->attn_ms += a;
  }
  out->n_layers = t->layers;
  out->launches = t->launches;
  return DD_OK;
}

dd_status dd_ctx_timings(dd_ctx* c, dd_phase_times* out) { return dd_ctx_step_timings(c, 0, out); }

dd_status dd_ctx_set_timing_depth(dd_ctx* c, int depth) {
  if (!c || depth < 1 || depth > kMaxTimingDepth) return DD_ERR_INVALID_ARG;
  for (size_t i = (size_t)depth; i < c->tsets.size(); ++i) c->tsets[i].release();
  c->tsets.resize((size_t)depth);
  c->t_depth = depth;
  c->t_last = -1;
  c->t_count = 0;
  return DD_OK;
}

dd_status dd_ctx_correction_stats(dd_ctx* c, int32_t* misses, float* mass, int n_layers) {
  if (!c || n_layers < 0) return DD_ERR_INVALID_ARG;
  if (c->last_corr_layers <= 0 || n_layers > c->last_corr_layers) return DD_ERR_INVALID_ARG;
  if (cudaEventSynchronize(c->ev_done) != cudaSuccess) return DD_ERR_CUDA;
  const size_t U = (size_t)c->dims.U;
  if (misses && cudaMemcpy(misses, c->miss, (size_t)n_layers * U * sizeof(int32_t),
                           cudaMemcpyDeviceToHost) != cudaSuccess)
    return DD_ERR_CUDA;
  if (mass && cudaMemcpy(mass, c->mass, (size_t)n_layers * U * 2 * sizeof(float),
                         cudaMemcpyDeviceToHost) != cudaSuccess)
    return DD_ERR_CUDA;
  return DD_OK;
}

dd_status dd_ctx_step_score_times(dd_ctx* c, int back, float* out_ms, int n) {
  if (!c || !out_ms || n < 0) return DD_ERR_INVALID_ARG;
  TimingSet* t = timing_set(c, back);
  if (!t) return DD_ERR_INVALID_ARG;
  for (int l = 0; l < t->layers && l < n; ++l) {
    const cudaEvent_t* e = &t->tev[(size_t)l * PH_N];
    if (cudaEventElapsedTime(&out_ms[l], e[PH_SCORE0], e[PH_SCORE1]) != cudaSuccess)
      return DD_ERR_CUDA;
  }
  return DD_OK;
}

dd_status dd_ctx_score_times(dd_ctx* c, float* out_ms, int n) {
  return dd_ctx_step_score_times(c, 0, out_ms, n);
}

}  // extern "C"
