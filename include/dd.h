/*
 * dd.h -- C ABI of libdd.so: the predictive sparse-KV decode step on one GB300
 * (sm_103a).
 *
 * The operation is the one the DualDecoder paper ("DualDecoder: Accelerate
 * Long Context LLM Inference by Predictive Prefetch", arXiv:2607.26475)
 * describes.  For each layer and each (request b, KV head h_kv), the library:
 *   1. scores the speculated token's query against the key cache,
 *      alpha = softmax(q_spec K^T / sqrt(d_k))
 *      (summary page of the paper, "core formulas"; paper Sec. 1: the
 *      retrieval index is computed from the token being processed);
 *   2. selects the per-head top-k entries, I = argtopk(alpha, k)
 *      (same formula; paper Fig. 1 "Select Top-k");
 *   3. gathers only the selected K/V rows from a pinned host-memory KV store
 *      into a layer-scoped GPU buffer (paper Sec. 2.2 and Fig. 1 "Sparse KV
 *      Gather"; summary page worked example, step 5);
 *   4. runs decode attention for the real query over the gathered rows plus a
 *      local window of the most recent W positions (paper Fig. 1 "Attention");
 *   5. loops over layers on two streams so that the gather of layer l+1
 *      overlaps the attention of layer l, through a double-buffered scratch
 *      region of O(k*d) bytes (paper Sec. 1: layer-aware transfer schedule and
 *      layer-scoped memory manager; summary page, memory formula O(n*d) ->
 *      O(k*d)).
 *
 * Conventions (every call):
 *  - Element type: DD_F32 (IEEE binary32) or DD_BF16 (bfloat16) for q_spec, q,
 *    K and V; all arithmetic accumulates in fp32; outputs are fp32.
 *  - Layouts are dense row-major, units are (b, h_kv) with u = b*H_kv + h_kv:
 *      q_spec, q        [B][H_q][d]
 *      K (device)       [B][H_kv][n][d]     the layer's full key cache in HBM
 *      K, V (host)      [B][H_kv][n][d]     pinned host store of the layer
 *      V window         [B][H_kv][W][d]     device copy of V rows [n-W, n)
 *      idx              [B][H_kv][k] int32  ascending positions in [0, n-W)
 *      sel_score        [B][H_kv][k] fp32   alpha (MHA) or group sum of alpha
 *      lse              [B][H_q]     fp32   log sum_j exp(s_j) over all n
 *      k_buf, v_buf     [B][H_kv][k][d]     gathered rows, in idx order
 *      out              [B][H_q][d]  fp32
 *    Query head h uses KV head h / (H_q / H_kv) (grouped-query attention).
 *  - Supported: head_dim 64 or 128 (fp32) and 64, 128 or 256 (bf16);
 *    H_q % H_kv == 0; 1 <= k <= n - W; 0 <= W < n.  Other shapes return
 *    DD_ERR_UNSUPPORTED or DD_ERR_INVALID_ARG.
 *  - Device pointers must be 16-byte aligned and belong to the current CUDA
 *    device (for dd_decode_step, the device the context was created on; the
 *    call is rejected on any other); host KV pointers must come from
 *    cudaHostAlloc / cudaMallocHost / cudaHostRegister (page-locked, mapped
 *    under unified addressing); pageable host memory is rejected.
 *  - Ownership: the caller owns every buffer passed in; the library never
 *    frees or retains them.  A dd_ctx owns only its scratch slots, its
 *    workspace and its events.
 *  - Synchronisation: calls enqueue work on the given stream(s) and return
 *    without synchronising.  Argument errors are reported synchronously
 *    (nothing is enqueued); a launch failure returns DD_ERR_CUDA; faults
 *    during execution surface at the caller's next synchronisation.
 *  - Threads: the per-layer calls may be made from any thread; a dd_ctx is
 *    used by one thread at a time (its steps share its scratch slots, events
 *    and workspace, so steps of one context must also not run concurrently
 *    on unrelated streams).
 *  - No exceptions cross this boundary.  The library has no CPU fallback.
 */
#ifndef DD_H
#define DD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DD_OK = 0,
  DD_ERR_INVALID_ARG = 1, /* null/misaligned/pageable pointer, inconsistent sizes */
  DD_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set */
  DD_ERR_OOM = 3,         /* device allocation failed (dd_ctx_create only) */
  DD_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  DD_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (dd_check_device) */
} dd_status;

typedef enum { DD_F32 = 0, DD_BF16 = 1 } dd_dtype;

/* One layer's shape. */
typedef struct {
  int32_t batch;      /* B: concurrent requests */
  int32_t n_q_heads;  /* H_q */
  int32_t n_kv_heads; /* H_kv (divides H_q) */
  int32_t head_dim;   /* d */
  int32_t ctx_len;    /* n: cached positions */
  int32_t top_k;      /* k: rows selected per (request, KV head) */
  int32_t window;     /* W: most recent positions always attended */
  int32_t dtype;      /* dd_dtype of q_spec, q, K, V */
} dd_shape;

/* Same handle type as cudaStream_t. */
typedef struct CUstream_st* dd_stream_t;

/* Static description of a status code; never NULL. */
const char* dd_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dd_version(void);

/*
 * Every wait inside the library's kernels (on an mbarrier that a bulk copy
 * completes) is bounded: after 2 s the kernel records the timeout in a
 * device-side status word, lets its copies in flight land and returns, so the
 * context stays usable.  This call synchronises the current device, returns
 * DD_ERR_TIMEOUT if any wait gave up since the previous call (DD_ERR_CUDA if
 * the device reports an error) and clears the status words.
 */
dd_status dd_check_device(void);

/*
 * Host KV store allocation.  The GPU reads the host store through the host's
 * page tables.  On a Grace host with 64 KiB base pages a long-context gather
 * touches hundreds of thousands of distinct pages per layer, each needing its
 * own translation; the translations slow the gather and the kernels running
 * beside it.  Huge pages cut them to a handful per layer.  dd_host_alloc maps
 * `bytes` (rounded up to whole huge pages) of anonymous memory aligned to the
 * host's huge-page size, asks for transparent huge pages (madvise), faults it
 * in from the CPU (several threads; the pages read as zero), locks it (mlock,
 * best effort: dd_host_store_locked reports whether it held) and registers it
 * with CUDA (cudaHostRegister).  The caller owns the memory, fills it from the
 * CPU and releases it with dd_host_free.  Returns DD_ERR_OOM if the mapping
 * fails and DD_ERR_CUDA if registration fails.  Any page-locked memory works
 * with the gather.
 * Measured on GB300 (512 MiB huge pages, a 64 GiB store filled and cycled by
 * gathers): when the host leaves it alone the gather holds 183-188 GB/s.  On
 * many freshly started hosts, though, the host split some of its huge pages
 * and migrated pages soon after the store was filled (by CPU writes or by
 * device-to-host copies alike, locked or not), and gathers then ran at
 * 1-10 GB/s for minutes; dd_host_alloc_pinned is the stable alternative.
 */
dd_status dd_host_alloc(size_t bytes, void** out);
/*
 * Host KV store in page-locked memory that the CUDA driver allocates
 * (cudaHostAlloc, portable), exactly `bytes`, in the host's base pages.  It
 * is the stable choice: on GB300 hosts the huge-page store of dd_host_alloc
 * gathers faster (183-188 against 131-176 GB/s on the GQA-128K layer) but
 * was, in most runs on freshly started hosts, split and moved by the host
 * shortly after it was filled, and its gathers then ran at 1-10 GB/s for
 * minutes; stores from this call never did.  Contents start undefined.
 * Released with dd_host_free.  DD_ERR_OOM if the allocation fails.
 */
dd_status dd_host_alloc_pinned(size_t bytes, void** out);
/* Release a region from dd_host_alloc (unlock, unregister, unmap) or
 * dd_host_alloc_pinned (NULL is a no-op); DD_ERR_INVALID_ARG for any other
 * pointer. */
dd_status dd_host_free(void* p);
/* 1 if p lies in a store from dd_host_alloc, 2 if from dd_host_alloc_pinned,
 * else 0. */
int dd_host_store_kind(const void* p);
/* 1 if p lies in a store from dd_host_alloc whose pages are locked, else 0. */
int dd_host_store_locked(const void* p);
/* The host huge-page size the allocator and the gather's translation
 * prefetch use (transparent-huge-page size, else 2 MiB). */
size_t dd_host_page_bytes(void);

/*
 * Bytes of device workspace that dd_score_topk, dd_sparse_decode_attn and
 * dd_correct_misses need for this shape (fp32 logits [B][H_q][round_up(n,4)],
 * per-chunk softmax partials, split-k attention partials, the real query's
 * selection scores and B*H_kv counters of the fused selection, each region
 * 256-byte aligned).  The calls use disjoint parts, so one buffer serves them
 * all (but two calls in flight at once need two buffers).
 * Returns DD_ERR_INVALID_ARG / DD_ERR_UNSUPPORTED for bad shapes.
 */
dd_status dd_workspace_size(const dd_shape* shape, size_t* bytes);

/*
 * How dd_score_topk (and the layer loop) computes this shape's logits: 1 if
 * on the tensor cores (bf16 keys with at least two query heads per KV head:
 * warp-level mma on 16-row key tiles, fp32 accumulation), 0 if in the
 * per-lane form (fp32 FMAs; single heads and fp32 keys).  Both give the
 * logits within the fp32 rounding bound of a d-term dot product.  Returns
 * -DD_ERR_INVALID_ARG or -DD_ERR_UNSUPPORTED for a bad shape.
 */
int dd_score_tensor_cores(const dd_shape* shape);

/*
 * Steps 1-2 for one layer: logits s[b,h,j] = q_spec[b,h] . K[b,h_kv(h),j] /
 * sqrt(d) for all j < n; lse_out[b,h] = log sum_j exp(s[b,h,j]); selection
 * score a[j] = exp(s_j - lse) (MHA) or sum over the query heads of the group
 * of exp(s_hj - lse_h) (GQA); idx_out = the k positions of [0, n-W) with the
 * largest a, ties to the lower position, written in ascending order, and
 * sel_score_out = a at those positions.
 *   q_spec   device [B][H_q][d]            k_dev  device [B][H_kv][n][d]
 *   idx_out  device [B][H_kv][k] int32     sel_score_out device [B][H_kv][k]
 *   lse_out  device [B][H_q] fp32 (may be NULL)
 *   workspace device, at least dd_workspace_size bytes.
 * Passage: summary page, core formulas (alpha = softmax(q_spec K^T /
 * sqrt(d_k)), I = argtopk(alpha, k)) and worked example, step 4; paper Sec. 1
 * (the retrieval index comes from the token being processed and the key
 * state); paper Fig. 1 "Select Top-k".
 */
dd_status dd_score_topk(const dd_shape* shape, const void* q_spec, const void* k_dev,
                        int32_t* idx_out, float* sel_score_out, float* lse_out, void* workspace,
                        size_t ws_bytes, dd_stream_t stream);

/*
 * Step 3 for one layer: for every unit u and slot i < k, copy row
 * idx[u][i] of the pinned host K and V stores into row i of k_buf / v_buf.
 * The rows are read by the GPU directly from page-locked host memory through
 * unified addressing, over the host link (zero-copy).
 *   k_host, v_host  pinned host [B][H_kv][n][d]
 *   idx             device [B][H_kv][k] int32, each in [0, n); an index
 *                   outside that range is clamped into it on the device, so
 *                   the kernel never reads outside the store
 *   k_buf, v_buf    device [B][H_kv][k][d]
 *   If a store was allocated by dd_host_alloc (huge pages), one warp first
 *   reads a word per huge page of the two host regions so their address
 *   translations are resolved once (a second, tiny kernel on the same stream).
 *   mode            0 = bulk-copy gather: one-warp CTAs issue one
 *                       cp.async.bulk per row into shared memory and write
 *                       tiles back with bulk stores (used by dd_decode_step);
 *                   1 = load/store gather: 16-byte loads from every thread
 *                       (the gathered rows of one tensor, B*H_kv*k*d
 *                       elements, below 8 GiB, else DD_ERR_UNSUPPORTED);
 *                   other values return DD_ERR_UNSUPPORTED.  Both modes give
 *                   identical bytes.  (Neither is a batched copy-engine
 *                   copy: one copy-engine request per 256-byte row would be
 *                   bound by its submission cost, and the one-call batched
 *                   copy routines are not used by this library.)
 * Passage: paper Sec. 2.2 (the host link is far slower than HBM and the
 * selected entries are scattered over the context, so only they are fetched);
 * paper Fig. 1 "Sparse KV Gather"; summary page worked example, step 5 (about
 * 2 MB per layer and request for LLaMA-2-7B at 32K with the top 128).
 */
dd_status dd_gather_h2d(const dd_shape* shape, const void* k_host, const void* v_host,
                        const int32_t* idx, void* k_buf, void* v_buf, int mode,
                        dd_stream_t stream);

/*
 * Step 3 from one interleaved host store: kv_host is pinned host memory laid
 * out [B][H_kv][n][2][d], each position's K row followed by its V row.
 * Otherwise as dd_gather_h2d, with identical bytes gathered.  A position's
 * two rows share a host page, so a gather over small pages needs fewer page
 * translations than over separate K and V stores: 12 % fewer for the GQA-128K
 * layer, 38 % fewer for the 7B-32K one with 64 KiB pages.
 * Passage: as dd_gather_h2d; the interleaved layout is this design's.
 */
dd_status dd_gather_h2d_kv(const dd_shape* shape, const void* kv_host, const int32_t* idx,
                           void* k_buf, void* v_buf, int mode, dd_stream_t stream);

/*
 * Geometry of the bulk-copy gather (mode 0) for every later launch in the
 * process, by dd_gather_h2d and dd_decode_step alike: grid_pct one-warp CTAs
 * per 100 SMs (1..800), tile_bytes of rows per tensor and shared-memory stage
 * (a multiple of 512, 512..16384; rows wider than a tile move one per stage),
 * and `stages` stages per CTA (1..8), with 2 * stages * tile_bytes at most
 * 227 KiB of shared memory.  Rows in flight are the CTAs times the
 * stages times the rows of a tile.  The default, (100, 4096, 3), puts one
 * 24 KiB CTA on each SM, which fits beside three scoring CTAs.  Launches
 * already enqueued keep the geometry they had.  DD_ERR_INVALID_ARG outside
 * the ranges.  The bytes gathered never depend on it.
 */
dd_status dd_set_gather_geometry(int grid_pct, int tile_bytes, int stages);
/*
 * Geometry of the load/store gather (mode 1) for every later launch in the
 * process: grid_pct CTAs per 100 SMs (1..800) of `threads` threads (a multiple
 * of 32, 32..256), each thread with 8 16-byte loads in flight.  The default is
 * (100, 256).  DD_ERR_INVALID_ARG outside the ranges.  The bytes gathered
 * never depend on it.
 */
dd_status dd_set_gather_lsu_geometry(int grid_pct, int threads);

/*
 * Step 4 for one layer: out[b,h] = sum_{j in S} softmax_S(q[b,h] . K_j /
 * sqrt(d)) V_j with S = the k gathered rows followed by the W window rows
 * [n-W, n).  Gathered rows come from k_buf / v_buf, window keys from k_dev
 * (rows [n-W, n) of each unit) and window values from v_win.  Split-k over
 * the k+W rows with a log-sum-exp merge of the partials (in workspace).
 *   q      device [B][H_q][d]        k_buf, v_buf device [B][H_kv][k][d]
 *   k_dev  device [B][H_kv][n][d]    v_win device [B][H_kv][W][d] (NULL if W=0)
 *   out    device [B][H_q][d] fp32
 * Passage: paper Fig. 1 "Attention" (decode attention over the fetched sparse
 * KV entries); paper Sec. 2.1 (attention of the current query over the cached
 * keys and values); summary page worked example, step 7 (the prefetched
 * entries serve the decoding step).
 */
dd_status dd_sparse_decode_attn(const dd_shape* shape, const void* q, const void* k_buf,
                                const void* v_buf, const void* k_dev, const void* v_win,
                                float* out, void* workspace, size_t ws_bytes,
                                dd_stream_t stream);

/*
 * The paper has no counterpart to this call.  It is dd_sparse_decode_attn
 * without the workspace argument, for callers that cannot allocate device
 * memory at all.  Examples: an engine that has already promised every free
 * byte of HBM to its KV-cache pool, or a plugin inside a framework that owns
 * all device allocations.  It also helps loops that must not stall the GPU:
 * cudaMalloc synchronises the device.  The call itself calls no allocator.
 *
 * The split-k partials live in one static device array of
 * DD_NOALLOC_SCRATCH_BYTES inside libdd.so.  Every GPU that loads the
 * library holds that array until the process exits.  A shape needs
 * round_up(B*H_q*S*d*4, 256) + B*H_q*S*8 bytes of it, where
 * S = ceil((k + W) / 64).  Larger shapes return DD_ERR_UNSUPPORTED and
 * enqueue nothing.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  That first call should
 * come before any stream capture.
 *
 * All calls share the array, and it keeps the last call's contents.  Nothing
 * in it needs to start at zero.  Calls that overlap on the GPU race on it, so
 * the caller must serialise them (one stream, or explicit ordering).
 * Arguments, layouts, results and errors are otherwise those of
 * dd_sparse_decode_attn.
 */
#define DD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
dd_status dd_sparse_decode_attn_noalloc(const dd_shape* shape, const void* q, const void* k_buf,
                                        const void* v_buf, const void* k_dev, const void* v_win,
                                        float* out, dd_stream_t stream);

/*
 * Miss correction for one layer, once the real query is known (paper Sec. 1:
 * the transfer schedule corrects prediction misses on the critical path;
 * summary page, weaknesses: a misprediction falls back to synchronous
 * retrieval).  Computes the real query's top-k exactly as dd_score_topk does
 * (idx_true_out, ascending), then writes its rows to k_buf_out / v_buf_out in
 * idx_true order: a row already in the prefetched buffers (idx_spec, k_buf_spec,
 * v_buf_spec, as left by dd_score_topk and dd_gather_h2d with the speculated
 * query) is copied on the device, a missed row is read from the pinned host
 * store.  miss_out[u] (optional) counts the missed rows of unit u; mass_out
 * (optional) is [B*H_kv][2]: the real query's selection score (alpha, or its
 * group sum) over the rows that were prefetched, and over all k rows.
 *   q            device [B][H_q][d]      the real query
 *   idx_spec     device [B][H_kv][k]     ascending, from the prediction
 *   k_buf_spec, v_buf_spec device [B][H_kv][k][d]
 *   k_host, v_host pinned host [B][H_kv][n][d]
 *   idx_true_out device [B][H_kv][k] int32
 *   k_buf_out, v_buf_out device [B][H_kv][k][d] (must not alias the inputs)
 * k above 4096 returns DD_ERR_UNSUPPORTED.  Uses the workspace of
 * dd_workspace_size.
 */
dd_status dd_correct_misses(const dd_shape* shape, const void* q, const void* k_dev,
                            const int32_t* idx_spec, const void* k_buf_spec,
                            const void* v_buf_spec, const void* k_host, const void* v_host,
                            int32_t* idx_true_out, void* k_buf_out, void* v_buf_out,
                            int32_t* miss_out, float* mass_out, void* workspace, size_t ws_bytes,
                            dd_stream_t stream);
/* dd_correct_misses with the rows the prediction missed read from one
 * interleaved host store [B][H_kv][n][2][d] (see dd_gather_h2d_kv). */
dd_status dd_correct_misses_kv(const dd_shape* shape, const void* q, const void* k_dev,
                               const int32_t* idx_spec, const void* k_buf_spec,
                               const void* v_buf_spec, const void* kv_host,
                               int32_t* idx_true_out, void* k_buf_out, void* v_buf_out,
                               int32_t* miss_out, float* mass_out, void* workspace,
                               size_t ws_bytes, dd_stream_t stream);

/*
 * Test hook (no counterpart in the paper): enqueue on `stream` a wait that
 * nothing completes; it gives up after limit_ns (1 ns .. 100 ms) through the
 * same bounded-wait path every kernel of the library uses, and the next
 * dd_check_device returns DD_ERR_TIMEOUT.  The kernel returns normally, so
 * the context stays usable.
 */
dd_status dd_debug_expire_wait(uint64_t limit_ns, dd_stream_t stream);

/* ------------------------ landmark selection ------------------------ */

/*
 * Chunk landmarks (DualDecoder paper, Sec. 1: the retrieval index is computed
 * from the current token and static GPU-resident KV landmarks; Sec. 2.2:
 * adjacent KV entries are grouped into chunks with compressed landmarks, the
 * GPU picks chunks for the current query and fetches their entries from host
 * memory).  The paper does not define the landmark; here it is the mean key
 * of each chunk of c adjacent positions of [0, n - W), in fp32:
 *   landmarks[u][m][t] = (1/c) sum_{r<c} K[u][m c + r][t],  M = (n - W) / c.
 * Constraints: c >= 2, c divides n - W and k, d in {64, 128}; otherwise
 * DD_ERR_UNSUPPORTED.
 */
dd_status dd_landmarks_size(const dd_shape* shape, int chunk, size_t* bytes);

/*
 * Build the landmarks of one layer's keys (device k_dev [B][H_kv][n][d] of the
 * shape's dtype) into device landmarks_out [B][H_kv][M][d] fp32.  Built once
 * per prefill: the keys of [0, n - W) do not change while decoding.
 */
dd_status dd_build_landmarks(const dd_shape* shape, int chunk, const void* k_dev,
                             float* landmarks_out, dd_stream_t stream);

/*
 * Landmark selection: score q_spec against the M landmarks exactly as
 * dd_score_topk scores keys (fp32 arithmetic; bf16 queries are widened first),
 * with no window, take each unit's top k/c chunks (ties to the lower chunk,
 * ascending), and write their k rows in ascending order:
 *   idx_out          device [B][H_kv][k] int32, chunk m -> rows m c .. m c + c - 1
 *   chunk_score_out  device [B][H_kv][k/c] f32, the chunk's selection score
 *                    (softmax over chunks, summed over the group's heads)
 *   lse_out          device [B][H_q] f32 over the chunk logits, or NULL
 * The workspace must hold dd_landmarks_workspace_size bytes.
 */
dd_status dd_landmarks_workspace_size(const dd_shape* shape, int chunk, size_t* bytes);
dd_status dd_score_topk_landmarks(const dd_shape* shape, int chunk, const void* q_spec,
                                  const float* landmarks, int32_t* idx_out, float* chunk_score_out,
                                  float* lse_out, void* workspace, size_t ws_bytes,
                                  dd_stream_t stream);

/* ---------------------------- layer loop ---------------------------- */

typedef struct dd_ctx dd_ctx;

/* Per-layer inputs and output of dd_decode_step (pointers as above). */
typedef struct {
  const void* q_spec; /* device [B][H_q][d] */
  const void* q;      /* device [B][H_q][d] */
  const void* k_dev;  /* device [B][H_kv][n][d] (see k_win) */
  const void* k_host; /* pinned host [B][H_kv][n][d] */
  const void* v_host; /* pinned host [B][H_kv][n][d] */
  const void* v_win;  /* device [B][H_kv][W][d] (NULL if W = 0) */
  float* out;         /* device [B][H_q][d] */
  const float* landmarks; /* device [B][H_kv][(n-W)/c][d] fp32 from dd_build_landmarks;
                             read only under DD_STEP_LANDMARKS (else may be NULL) */
  const void* k_win;  /* device [B][H_kv][W][d], the window's keys, or NULL: then
                         they are read from k_dev.  Under DD_STEP_LANDMARKS with
                         k_win (or W = 0) k_dev may be NULL: nothing of size n
                         then stays on the device */
  const void* kv_host; /* pinned host [B][H_kv][n][2][d]: one store holding each
                          position's K row followed by its V row, in place of
                          k_host and v_host (which must then be NULL); NULL to
                          use k_host and v_host.  See dd_gather_h2d_kv */
} dd_layer_io;

/*
 * Allocate the layer-scoped state for one shape: two scratch slots of
 * gathered K/V rows (2 x 2 x B*H_kv*k*d elements; independent of n), two index
 * slots, the workspace and the events.  Returns DD_ERR_OOM on allocation
 * failure.  Uses the current CUDA device; the context is bound to it.  The
 * number of layers is not fixed here: each dd_decode_step passes its own
 * layer list, and the per-layer state is what the two slots hold.
 */
dd_status dd_ctx_create(const dd_shape* shape, dd_ctx** out);
void dd_ctx_destroy(dd_ctx* ctx);

/* Bytes of device memory a context holds: the two layer slots (gathered K
 * and V rows, 2 x 2 x B*H_kv*k*d elements; their indices and selection
 * scores, 2 x 2 x B*H_kv*k x 4 bytes), the query heads' LSE (B*H_q x 4 bytes)
 * and the workspace (dd_workspace_size; its fp32 logits, 4 bytes per query
 * head and position, are the only part that grows with n), plus the
 * miss-correction and landmark buffers once those are used. */
size_t dd_ctx_device_bytes(const dd_ctx* ctx);

enum {
  DD_STEP_TIMING = 1,     /* record per-phase CUDA events; read with dd_ctx_timings */
  DD_STEP_LATE_GATHER = 2, /* start the gather of layer l+1 after the attention of
                              layer l (it then overlaps the scoring of layer l+2) */
  DD_STEP_GATHER_LSU = 4,  /* gather with dd_gather_h2d mode 1 (load/store)
                              instead of mode 0 (bulk copy) */
  DD_STEP_CORRECT_MISSES = 16, /* before each layer's attention, compute the
                              real query's own top-k and attend over exactly those
                              rows, fetching the ones the prediction missed
                              (dd_correct_misses; k <= 4096; not combinable with
                              DD_STEP_PIPELINE); statistics via
                              dd_ctx_correction_stats */
  DD_STEP_PIPELINE = 8,    /* two-stage pipeline: scoring and top-k of every
                              layer on `compute`; the gather and then the
                              attention of each layer on `copy`, as soon as its
                              indices are ready (compute runs at most two layers
                              ahead); attention never runs beside a gather */
  DD_STEP_TIMING_LIGHT = 64, /* like DD_STEP_TIMING, but only the step's first
                              and last events and those around each layer's
                              scoring (selection) phase; dd_ctx_timings then
                              reports step_ms and score_ms only */
  DD_STEP_FUSED_TOPK = 128, /* one kernel for steps 1-2: the scoring kernel's
                              last CTA of each unit selects that unit's rows
                              (no separate top-k launch; same results).  Off by
                              default: on GB300 the two-kernel form measured
                              faster on the MHA and GQA workloads */
  DD_STEP_GATHER_BESIDE_ATTN = 256,   /* overlapped schedule in which the scoring
                                         of layer l+1 waits for the gather of layer
                                         l: each gather overlaps only the previous
                                         layer's attention, never a scoring kernel */
  DD_STEP_DEBUG_DELAY_COPY = 512,     /* test hook: a 50 us GPU sleep before each
                                         gather, on the stream that runs it */
  DD_STEP_DEBUG_DELAY_COMPUTE = 1024, /* test hook: the same before each attention;
                                         with either, results must not change */
  DD_STEP_LANDMARKS = 32   /* select with dd_score_topk_landmarks over each
                              layer's `landmarks` instead of scoring every key
                              (chunk set by dd_ctx_set_landmark_chunk; not
                              combinable with DD_STEP_CORRECT_MISSES) */
};

/*
 * Landmark chunk size for DD_STEP_LANDMARKS.  Allocates the context's landmark
 * workspace on first use (or when a larger one is needed; then it first waits
 * for the device).  Same constraints as dd_score_topk_landmarks.
 */
dd_status dd_ctx_set_landmark_chunk(dd_ctx* ctx, int chunk);

/*
 * Enqueue one decode step over n_layers layers.  Steps 1-2 of layer l+1 run
 * on `compute` ahead of the attention of layer l; the gather of layer l+1 runs
 * on `copy` into the other scratch slot while layer l's attention runs.
 * Events order each gather after its indices and after the attention that
 * last read its slot, and each attention after its gather.  The copy stream
 * is joined back into `compute` before return.  If copy == compute (or copy
 * is NULL) every phase runs in order on `compute` (the serial schedule, with
 * bit-identical results).  Flags that choose a schedule other than the
 * pipeline (DD_STEP_LATE_GATHER, DD_STEP_GATHER_BESIDE_ATTN) together with
 * DD_STEP_PIPELINE return DD_ERR_UNSUPPORTED; in the serial schedule every
 * phase already runs alone, so they have no effect there.
 * Per-phase times are read afterwards with dd_ctx_timings (flags
 * DD_STEP_TIMING / DD_STEP_TIMING_LIGHT) instead of an output array, so that
 * steps can be enqueued back to back without a host wait.
 * Passage: paper Sec. 1 (layer-aware transfer schedule; layer-scoped KV memory
 * manager); summary page, core formulas (T_transfer = sum_l S_l / B hidden by
 * min max(T_compute, T_transfer); buffer O(n d) -> O(k d)) and worked example,
 * step 6 (the transfer overlaps the attention of other layers).
 */
dd_status dd_decode_step(dd_ctx* ctx, const dd_layer_io* layers, int n_layers,
                         dd_stream_t compute, dd_stream_t copy, int flags);

/*
 * Capture one decode step (same arguments as dd_decode_step, without the
 * timing flags) into a CUDA graph held by the context, replacing any earlier
 * one.  The step is first run once directly on `compute` (and synchronised),
 * so that everything it allocates lazily exists, then captured from
 * `compute` (the copy stream joins the capture through the step's events).
 * The graph keeps the layer pointers it was captured with: capture again when
 * they change.  DD_ERR_UNSUPPORTED with timing flags.
 */
dd_status dd_ctx_capture_step(dd_ctx* ctx, const dd_layer_io* layers, int n_layers,
                              dd_stream_t compute, dd_stream_t copy, int flags);

/* Launch the captured step on `stream` (one graph launch: the whole step,
 * both streams' work, with the same ordering as dd_decode_step). */
dd_status dd_ctx_replay_step(dd_ctx* ctx, dd_stream_t stream);

/* Phase times of the last dd_decode_step run with DD_STEP_TIMING, in ms. */
typedef struct {
  float step_ms;      /* first event to last event on `compute` */
  float score_ms;     /* sum over layers of the scoring kernel */
  float topk_ms;      /* sum over layers of LSE merge + top-k */
  float gather_ms;    /* sum over layers of the gather */
  float attn_ms;      /* sum over layers of attention (+ merge) */
  int32_t n_layers;
  int32_t launches;   /* kernels launched by that step */
} dd_phase_times;

/* Wait for the last timed step and read its phase times. */
dd_status dd_ctx_timings(dd_ctx* ctx, dd_phase_times* out);

/*
 * Keep the events of the last `depth` timed steps (1 <= depth <= 4096;
 * default 1), so that several timed steps can be enqueued back to back and
 * read afterwards.  Forgets the steps recorded so far.  Must not be called
 * while a timed step is being enqueued on another thread.
 */
dd_status dd_ctx_set_timing_depth(dd_ctx* ctx, int depth);

/* Phase times of the timed step `back` steps before the last one (0: the
 * last); waits for that step.  DD_ERR_INVALID_ARG if the ring no longer holds
 * it. */
dd_status dd_ctx_step_timings(dd_ctx* ctx, int back, dd_phase_times* out);

/*
 * Miss statistics of the last step run with DD_STEP_CORRECT_MISSES, for its
 * first n_layers layers (waits for that step): misses [n_layers][B*H_kv]
 * (rows of the real query's top-k that the prediction had not fetched) and
 * mass [n_layers][B*H_kv][2] (the real query's selection score summed over the
 * rows the prediction had fetched, and over all k rows).  Either may be NULL.
 */
dd_status dd_ctx_correction_stats(dd_ctx* ctx, int32_t* misses, float* mass, int n_layers);

/* Per-layer scoring-kernel times (ms) of the last timed step; n entries max.
 * Under DD_STEP_LANDMARKS the time covers the whole landmark selection. */
dd_status dd_ctx_score_times(dd_ctx* ctx, float* out_ms, int n);
/* The same for the timed step `back` steps before the last one. */
dd_status dd_ctx_step_score_times(dd_ctx* ctx, int back, float* out_ms, int n);

#ifdef __cplusplus
}
#endif
#endif /* DD_H */
