// Step 1 of the decode step: score the speculated token's query against the
// key cache, s[b,h,j] = q_spec[b,h] . K[b,h_kv,j] / sqrt(d), together with the
// online softmax statistics (max, sum of exp) of every chunk of positions.
// (DualDecoder summary page, core formulas: alpha = softmax(q_spec K^T /
// sqrt(d_k)); paper Sec. 1: the retrieval index is computed from the token
// being processed and the key cache.)
//
// The kernel is HBM-bound: every K row is read exactly once, 2 flops per
// element and query head.  Each CTA owns one chunk of positions of one
// (request, KV head) unit.  One producer warp streams the chunk through a
// ring of shared-memory stages with bulk copies (cp.async.bulk on the
// tensor-memory-access unit, completion on an mbarrier, K tagged L2
// evict-first), so many bytes are in flight per SM without occupying the
// load/store pipeline or registers.  Eight consumer warps read each stage:
// LPR lanes share one K row (16 bytes each), the dot products use packed fp32
// FMAs, the partial sums are reduced with a transposed xor-shuffle butterfly,
// and the lane that owns a row writes its logit and folds it into a running
// (max, sum of exp).  All query heads of a GQA group are scored from the same
// K row.  With FUSED, the unit's last CTA also runs its top-k (select.cuh).
//
// bf16 keys scored by a group of two or more query heads take the tensor
// cores instead: the group's heads times a 16-row tile of keys is a small
// matrix product (one column per head), which one warp-level mma per 16
// elements of the row computes with fp32 accumulation.  The FMA and widening
// instructions that make the per-lane form issue-bound for a GQA group
// disappear, and the issue slots they free serve the host gather running
// beside the scoring (see the consumer below).  A single head (MHA) keeps the
// per-lane form, which already streams at the copy rate; the tensor-core form
// handles it too (build option below) and measured no faster.
#include <math.h>

#include <type_traits>

#include "dd_internal.cuh"
#include "select.cuh"

namespace dd {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kScoreThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kStageBytes = 16384;
constexpr int kStages = 4;
// A CTA's chunk is 16 stages (256 KiB of K) when there is enough work; for
// small layers (few units, short rows, landmark caches) it shrinks by halves,
// down to the 4 stages of the ring, until the grid has kTargetCtas CTAs, so
// that the last wave of CTAs is a small share of the launch.
constexpr int kStagesPerChunk = 16;
constexpr int kMinStagesPerChunk = 4;
constexpr long long kTargetCtas = 4096;

// Set when a bounded wait gave up (read and cleared by dd_check_device).
__device__ unsigned int g_score_status = 0;

template <typename T, int D>
struct ScoreGeom {
  static constexpr int kVec = Elem<T>::kVec;            // elements per 16 bytes
  static constexpr int kRowBytes = D * (int)sizeof(T);  // 128, 256 or 512
  static constexpr int kLpr = D / kVec;                 // lanes per row
  static constexpr int kRpw = 32 / kLpr;                // rows per warp per pass
  static constexpr int kGroups = kConsumerWarps * kRpw; // row groups per CTA
  static constexpr int kStageRows = kStageBytes / kRowBytes;
  static constexpr int kRowsPerGroup = kStageRows / kGroups;
  static constexpr int kChunk = kStageRows * kStagesPerChunk;  // rows, at most
  static constexpr int kMinChunk = kStageRows * kMinStagesPerChunk;
  static_assert(kLpr >= kRowsPerGroup && kLpr <= 32, "unsupported row width");
  static_assert(kStageRows % kGroups == 0, "stage must hold whole row groups");
};

// Whether a layout is scored on the tensor cores: bf16 keys and query, and
// at least DD_SCORE_MMA_MIN_GROUP query heads per KV head (a build option:
// 1 sends MHA layers to the tensor cores as well).
#ifndef DD_SCORE_MMA_MIN_GROUP
#define DD_SCORE_MMA_MIN_GROUP 2
#endif
template <typename T, int G, bool QB>
__host__ __device__ constexpr bool use_mma() {
  return std::is_same<T, bf16_t>::value && !QB && G >= DD_SCORE_MMA_MIN_GROUP;
}
// The tensor-core consumer reads each key row as four lanes' 16-byte pieces.
// Rows start on 128-byte bank boundaries, so two rows at the same piece meet
// in the same banks.  Its stages are therefore filled as two halves with the
// second 64 bytes further on: a warp's loads then always pair a row of one
// half with a row of the other and touch every bank once.
constexpr int kHalfSkew = 64;
template <bool MMA>
__host__ __device__ constexpr int stage_stride() {
  return MMA ? kStageBytes + kHalfSkew : kStageBytes;
}

// Fused selection: the last CTA of a unit to finish runs the unit's top-k
// with its eight consumer warps, reusing the ring's shared memory.
constexpr int kSelWarps = kConsumerWarps;
constexpr int kSelCap = 1024;  // list entries per warp
using SelSmem = sel::Smem<kSelWarps, kSelCap>;
template <bool MMA>
__host__ __device__ constexpr size_t ring_bytes() {
  return (size_t)kStages * stage_stride<MMA>();
}
// Dynamic shared memory: [0, region): the ring (and, when FUSED, later the
// selection's lists, which need more); then the mbarriers.  The plain kernel
// asks only for the ring, so that three of its CTAs leave room on an SM for a
// gather CTA running beside them.
template <bool FUSED, bool MMA>
__host__ __device__ constexpr size_t region_bytes() {
  return ((FUSED && sizeof(SelSmem) > ring_bytes<MMA>() ? sizeof(SelSmem) : ring_bytes<MMA>()) +
          127) / 128 * 128;
}
template <bool FUSED, bool MMA>
__host__ __device__ constexpr size_t score_smem() {
  return region_bytes<FUSED, MMA>() + 2 * kStages * sizeof(uint64_t);
}

// D[16x8] += A[16x16] B[16x8] on the tensor cores, bf16 inputs, fp32
// accumulation.  Fragments (g = lane / 4, c = lane % 4): a0 = A[g][2c..2c+1],
// a1 = A[g+8][2c..2c+1], a2 = A[g][2c+8..2c+9], a3 = A[g+8][2c+8..2c+9];
// b0 = B[2c..2c+1][g], b1 = B[2c+8..2c+9][g]; d = D[g][2c..2c+1],
// D[g+8][2c..2c+1].  Each register holds two bf16, the lower k in the low half.
__device__ __forceinline__ void mma_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Fold logit sv into a running (max, sum of exp) with one exponential: a new
// maximum rescales the sum, any other logit adds its term.
__device__ __forceinline__ void online_lse(float sv, float& m_run, float& l_run) {
  const float dv = sv - m_run;
  const float ev = __expf(-fabsf(dv));
  l_run = dv > 0.f ? fmaf(l_run, ev, 1.f) : l_run + ev;
  m_run = fmaxf(m_run, sv);
}

// Selection outputs of the fused kernel (unused when FUSED is false).
struct FusedOut {
  int32_t* counters;  // [U], zero before the launch; each unit's last CTA re-zeroes its own
  int32_t* idx;       // [U][k]
  float* sel;         // [U][k]
  float* lse;         // [B][H_q] or NULL
  int span, k;
};

// QB: the keys are fp32 (landmarks) but the query is bf16; it is widened
// exactly on load.
template <typename T, int D, int G, bool FUSED, bool QB = false>
__global__ void __launch_bounds__(kScoreThreads, use_mma<T, G, QB>() && !FUSED ? 3 : 1)
    score_kernel(const uint4* __restrict__ q_spec, const unsigned char* __restrict__ K,
                 float* __restrict__ logits, float2* __restrict__ part, int n, int ldn, int Hq,
                 int Hkv, int chunk, int nchunks, float scale, FusedOut fo) {
  using Geo = ScoreGeom<T, D>;
  constexpr int VEC = Geo::kVec, LPR = Geo::kLpr, RPW = Geo::kRpw, NG = Geo::kGroups;
  constexpr int SR = Geo::kStageRows, RPG = Geo::kRowsPerGroup, RB = Geo::kRowBytes;
  constexpr int N = G * RPG;                     // partial sums per lane per stage
  constexpr int S = ilog2(N) < ilog2(LPR) ? ilog2(N) : ilog2(LPR);  // transposing steps
  constexpr int P = N >> S;                      // totals per lane after the reduction
  static_assert(P <= RPG && RPG % P == 0, "a lane's totals must share one head");
  constexpr bool MMA = use_mma<T, G, QB>();
  constexpr int STRIDE = stage_stride<MMA>();
  constexpr int HALF = SR / 2;  // rows in each half of a stage (tensor-core form)

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + region_bytes<FUSED, MMA>());
  uint64_t* empty = full + kStages;

  const int item = blockIdx.x;
  const int u = item / nchunks, c = item - u * nchunks;
  const int b = u / Hkv, hk = u - b * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j_begin = c * chunk;
  const int j_end = min(n, j_begin + chunk);
  const int n_stages = (j_end - j_begin + SR - 1) / SR;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // Running (max, sum of exp) of the logits this lane writes: heads head0
  // and, in the tensor-core form, head0 + 1 (head0 = -1: the lane writes none).
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  int head0 = -1;
  bool ok = true;
  const unsigned char* Ku = K + (size_t)u * n * RB;

  if (warp == kConsumerWarps) {
    // Producer: one lane keeps up to kStages bulk copies in flight.
    if (lane == 0) {
      // K is read once: its lines go first when L2 needs room, so the logits
      // written by this launch stay there for the selection that reads them.
      const uint64_t policy = l2_evict_first_policy();
      for (int t = 0; t < n_stages; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !mbar_wait(&empty[s], ((t / kStages) - 1) & 1)) {
          ok = false;
          break;
        }
        const int r0 = j_begin + t * SR;
        const int nr = min(SR, j_end - r0);
        unsigned char* dst = ring + (size_t)s * STRIDE;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * RB));
        if constexpr (MMA) {  // two halves, the second kHalfSkew bytes on
          const int na = min(nr, HALF);
          bulk_load_hint(dst, Ku + (size_t)r0 * RB, (uint32_t)(na * RB), &full[s], policy);
          if (nr > HALF)
            bulk_load_hint(dst + HALF * RB + kHalfSkew, Ku + (size_t)(r0 + HALF) * RB,
                           (uint32_t)((nr - HALF) * RB), &full[s], policy);
        } else {
          bulk_load_hint(dst, Ku + (size_t)r0 * RB, (uint32_t)(nr * RB), &full[s], policy);
        }
      }
    }
  } else if constexpr (MMA) {
    // Tensor-core consumer.  A stage is TPS tiles of 16 rows; tile tau holds
    // rows tau*8 .. tau*8+7 of each half, the even mma rows from the first
    // half and the odd ones from the second (mma row m: half m & 1, row
    // tau*8 + m/2), and the stage's tiles go to the warps in turn.  The mma's
    // A operand is the tile of keys, its B operand the group's query heads
    // (columns G..7 zero).  The contraction over the d elements of a row is
    // taken in blocks of 32: lane (g, c) loads the 16-byte piece c of block
    // bb of its rows g and g+8 (A) and of query head g (B), and both operands
    // map the eight elements of a piece to the same logical k of two mmas
    // (elements 0-1 -> k 2c..2c+1 and 2-3 -> k 2c+8..2c+9 of the first mma,
    // elements 4-7 likewise of the second), so every element of the row
    // meets its query element exactly once.
    constexpr int TPS = SR / 16;
    constexpr int NB = D / 32;
    static_assert(SR % 16 == 0 && TPS <= kConsumerWarps && kConsumerWarps % TPS == 0,
                  "a stage must split into whole tiles, at most one per warp");
    static_assert(RB % 128 == 0, "rows must start on bank boundaries");
    const int gq = lane >> 2, cq = lane & 3;
    uint4 qb[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb)
      qb[bb] = gq < G ? ld_ro(q_spec + (size_t)(b * Hq + hk * G + gq) * (D / 8) + 4 * bb + cq)
                      : make_uint4(0u, 0u, 0u, 0u);
    // Accumulator columns 2c and 2c+1 are heads 2c and 2c+1 (G is 1 or even).
    if (2 * cq < G) head0 = 2 * cq;
    constexpr bool kPair = G >= 2;  // does column 2c+1 hold a head as well?
    const int par = gq & 1, hr = gq >> 1;
    // Byte offsets in a stage of the lane's piece of rows g and g+8 of tile 0.
    const int off0 = (par ? HALF * RB + kHalfSkew : 0) + hr * RB + 16 * cq;
    const int off1 = off0 + 4 * RB;
    float* lg = logits + (size_t)(b * Hq + hk * G + (head0 < 0 ? 0 : head0)) * ldn;

    for (int t = 0; t < n_stages; ++t) {
      const int s = t % kStages;
      if (!mbar_wait(&full[s], (t / kStages) & 1)) {
        ok = false;
        break;
      }
      const int tau = warp - ((t * TPS) & (kConsumerWarps - 1));
      const bool mine = tau >= 0 && tau < TPS;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (mine) {
        const unsigned char* base = ring + (size_t)s * STRIDE + tau * 8 * RB;
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
          const uint4 a0 = *reinterpret_cast<const uint4*>(base + off0 + 64 * bb);
          const uint4 a1 = *reinterpret_cast<const uint4*>(base + off1 + 64 * bb);
          mma_16x8x16(acc, a0.x, a1.x, a0.y, a1.y, qb[bb].x, qb[bb].y);
          mma_16x8x16(acc, a0.z, a1.z, a0.w, a1.w, qb[bb].z, qb[bb].w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled
      if (mine && head0 >= 0) {
        const int j0 = j_begin + t * SR + par * HALF + tau * 8 + hr;  // mma row g
        const int j1 = j0 + 4;                                          // mma row g + 8
        if (j0 < j_end) {
          const float s0 = acc[0] * scale;
          lg[j0] = s0;
          online_lse(s0, m_run[0], l_run[0]);
          if (kPair) {
            const float s1 = acc[1] * scale;
            lg[ldn + j0] = s1;
            online_lse(s1, m_run[1], l_run[1]);
          }
        }
        if (j1 < j_end) {
          const float s2 = acc[2] * scale;
          lg[j1] = s2;
          online_lse(s2, m_run[0], l_run[0]);
          if (kPair) {
            const float s3 = acc[3] * scale;
            lg[ldn + j1] = s3;
            online_lse(s3, m_run[1], l_run[1]);
          }
        }
      }
    }
  } else {
    const int sub = lane % LPR;
    const int grp = warp * RPW + lane / LPR;
    // The lane's partial sums live in acc[N], N = G * RPG values (head g,
    // stage row slot i).  The transposed reduction below halves them S times,
    // each time keeping the lower half of the slots and sending the upper
    // half to the lane 2^t away.  For that to need no selects, each lane
    // stores value v in slot v ^ X: X has, at bit LOGN-1-t, bit t of `sub`,
    // so at step t the lane keeps exactly the values its side of the pair
    // owns.  The permutation costs nothing inside the loop: slot (g, i) is
    // computed from head g ^ Xg (the query is loaded permuted) and stage row
    // i ^ Xi (a per-lane shared-memory offset).  After the S steps, lane
    // `sub` holds the totals of the P values X + p (p < P); X = prefix * P
    // where prefix is `sub`'s low S bits reversed.  Only lanes with
    // sub < 2^S hold distinct values, and all of one lane's values belong to
    // the same head g_lane.
    constexpr int LOGN = ilog2(N);
    int X = 0;
#pragma unroll
    for (int t = 0; t < S; ++t) X |= ((sub >> t) & 1) << (LOGN - 1 - t);
    const int Xg = X / RPG, Xi = X % RPG;
    float qf[G][VEC];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const size_t piece = (size_t)(b * Hq + hk * G + (g ^ Xg)) * LPR + sub;
      if constexpr (QB) {
        static_assert(VEC == 4, "a bf16 query widens to fp32 keys only");
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(q_spec) + piece);
        qf[g][0] = __uint_as_float(v.x << 16);
        qf[g][1] = __uint_as_float(v.x & 0xFFFF0000u);
        qf[g][2] = __uint_as_float(v.y << 16);
        qf[g][3] = __uint_as_float(v.y & 0xFFFF0000u);
      } else {
        unpack(ld_ro(q_spec + piece), qf[g]);
      }
    }
    // Shared-memory offset (in 16-byte pieces) of the row in slot i.
    int row_off[RPG];
#pragma unroll
    for (int i = 0; i < RPG; ++i) row_off[i] = ((i ^ Xi) * NG + grp) * LPR + sub;

    const int prefix = X / P;
    const int g_lane = X / RPG;
    const bool writer = (sub >> S) == 0;
    if (writer) head0 = g_lane;
    float* lg_row = logits + (size_t)(b * Hq + hk * G + g_lane) * ldn;

    for (int t = 0; t < n_stages; ++t) {
      const int s = t % kStages;
      if (!mbar_wait(&full[s], (t / kStages) & 1)) {
        ok = false;
        break;
      }
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * STRIDE);
      const int r0 = j_begin + t * SR;
      // Stage row (i * NG + grp), for i < RPG, belongs to this lane group.
      float acc[N];
      static_assert(RPG % 2 == 0, "rows are summed in pairs");
#pragma unroll
      for (int i = 0; i < RPG; i += 2) {
        float k0[VEC], k1[VEC];
        unpack(st[row_off[i]], k0);
        unpack(st[row_off[i + 1]], k1);
        // Packed fp32 FMA (two lanes of arithmetic per instruction): the even
        // and the odd elements accumulate separately; one packed add then
        // finishes two rows' dot products.
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 qv = make_float2(qf[g][e], qf[g][e + 1]);
            a0 = __ffma2_rn(qv, make_float2(k0[e], k0[e + 1]), a0);
            a1 = __ffma2_rn(qv, make_float2(k1[e], k1[e + 1]), a1);
          }
          const float2 sum = __fadd2_rn(make_float2(a0.x, a1.x), make_float2(a0.y, a1.y));
          acc[g * RPG + i] = sum.x;
          acc[g * RPG + i + 1] = sum.y;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled
      // Transposed reduction over the LPR lanes of the group: at step t each
      // lane keeps the lower half of its slots, sends the upper half to the
      // lane 2^t away and adds what it receives.
#pragma unroll
      for (int t2 = 0; t2 < S; ++t2) {
        const int half = (N >> t2) / 2;
#pragma unroll
        for (int i = 0; i < half; ++i)
          acc[i] = acc[i] + __shfl_xor_sync(0xffffffffu, acc[i + half], 1 << t2);
      }
      // Remaining lane bits: plain butterfly on the P values left.
#pragma unroll
      for (int off = 1 << S; off < LPR; off <<= 1)
#pragma unroll
        for (int p = 0; p < P; ++p) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], off);
      if (writer) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const int i = (prefix * P + p) % RPG;
          const int j = r0 + i * NG + grp;
          if (j < j_end) {
            const float sv = acc[p] * scale;
            lg_row[j] = sv;
            online_lse(sv, m_run[0], l_run[0]);
          }
        }
      }
    }
  }
  if (!ok) atomicOr(&g_score_status, 1u);
  __syncthreads();
  if (!ok && threadIdx.x == 0) {
    // A wait gave up: let the copies still in flight land before exiting.
    for (int s = 0; s < kStages; ++s) {
      mbar_wait(&full[s], 0);
      mbar_wait(&full[s], 1);
    }
  }

  // CTA-wide merge of the (max, sum) pairs of each head.
  __shared__ float2 red[G][kConsumerWarps + 1];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float2 p = make_float2(-INFINITY, 0.f);
    if (head0 >= 0 && g == head0) p = make_float2(m_run[0], l_run[0]);
    if (MMA && G >= 2 && head0 >= 0 && g == head0 + 1) p = make_float2(m_run[1], l_run[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float2 o;
      o.x = __shfl_xor_sync(0xffffffffu, p.x, off);
      o.y = __shfl_xor_sync(0xffffffffu, p.y, off);
      p = lse_merge(p, o);
    }
    if (lane == 0) red[g][warp] = p;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float2 p = red[g][0];
#pragma unroll
    for (int w = 1; w <= kConsumerWarps; ++w) p = lse_merge(p, red[g][w]);
    part[(size_t)(u * G + g) * nchunks + c] = p;
  }
  if (!FUSED) return;

  // Fused selection.  Every thread fences its logits and (max, sum) pair,
  // then one thread counts the CTA in; the CTA that completes the unit's
  // count (all others have fenced and counted before) selects its top-k.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(fo.counters + u, 1) == nchunks - 1;
  __syncthreads();
  if (!s_last || warp == kConsumerWarps) return;  // the producer warp is not needed
  __threadfence();
  if (threadIdx.x == 0) fo.counters[u] = 0;  // ready for the next launch
  // Every bulk copy into the ring has landed (all stages were waited for), so
  // its memory can hold the selection's histogram and lists.
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem);
  sel::merge_lse<G, true>(part, u, b, hk, Hq, nchunks, fo.lse, sm);
  sel::sync<kSelWarps>();
  sel::select_unit<G, true>(sm, logits + (size_t)(b * Hq + hk * G) * ldn, ldn, fo.span, fo.k,
                            fo.idx + (size_t)u * fo.k, fo.sel + (size_t)u * fo.k);
}

template <typename T, int D, int G, bool FUSED, bool QB = false>
cudaError_t launch_typed(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, const FusedOut& fo, cudaStream_t st) {
  static unsigned long long prepared = 0;
  constexpr size_t smem_bytes = score_smem<FUSED, use_mma<T, G, QB>()>();
  cudaError_t e = prepare_kernel(score_kernel<T, D, G, FUSED, QB>, &prepared, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)d.d);
  const unsigned grid = (unsigned)d.U * (unsigned)d.nchunks;
  score_kernel<T, D, G, FUSED, QB><<<grid, kScoreThreads, smem_bytes, st>>>(
      static_cast<const uint4*>(q_spec), static_cast<const unsigned char*>(k_dev), logits, part,
      d.n, d.ldn, d.Hq, d.Hkv, d.chunk, d.nchunks, scale, fo);
  return cudaGetLastError();
}

template <typename T, int D, bool FUSED>
cudaError_t launch_g(const Dims& d, const void* q, const void* k, float* lg, float2* p,
                     const FusedOut& fo, cudaStream_t st) {
  switch (d.G) {
    case 1: return launch_typed<T, D, 1, FUSED>(d, q, k, lg, p, fo, st);
    case 2: return launch_typed<T, D, 2, FUSED>(d, q, k, lg, p, fo, st);
    case 4: return launch_typed<T, D, 4, FUSED>(d, q, k, lg, p, fo, st);
    case 8: return launch_typed<T, D, 8, FUSED>(d, q, k, lg, p, fo, st);
  }
  return cudaErrorInvalidValue;
}

template <bool FUSED>
cudaError_t launch_any(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                       float2* part, const FusedOut& fo, cudaStream_t st) {
  if (d.dtype == DD_BF16) {
    if (d.d == 64) return launch_g<bf16_t, 64, FUSED>(d, q_spec, k_dev, logits, part, fo, st);
    if (d.d == 128) return launch_g<bf16_t, 128, FUSED>(d, q_spec, k_dev, logits, part, fo, st);
    if (d.d == 256) return launch_g<bf16_t, 256, FUSED>(d, q_spec, k_dev, logits, part, fo, st);
  } else {
    if (d.d == 64) return launch_g<float, 64, FUSED>(d, q_spec, k_dev, logits, part, fo, st);
    if (d.d == 128) return launch_g<float, 128, FUSED>(d, q_spec, k_dev, logits, part, fo, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

namespace {
template <typename T, int D>
int chunk_for(long long units, int n) {
  int rows = ScoreGeom<T, D>::kChunk;
  while (rows > ScoreGeom<T, D>::kMinChunk && units * ((n + rows - 1) / rows) < kTargetCtas)
    rows /= 2;
  return rows;
}
}  // namespace

bool score_uses_mma(int dtype, int group) {
  return dtype == DD_BF16 && group >= DD_SCORE_MMA_MIN_GROUP;
}

int score_chunk(int dtype, int head_dim, long long units, int n) {
  if (dtype == DD_BF16) {
    if (head_dim == 64) return chunk_for<bf16_t, 64>(units, n);
    if (head_dim == 128) return chunk_for<bf16_t, 128>(units, n);
    if (head_dim == 256) return chunk_for<bf16_t, 256>(units, n);
  } else {
    if (head_dim == 64) return chunk_for<float, 64>(units, n);
    if (head_dim == 128) return chunk_for<float, 128>(units, n);
  }
  return 0;
}

cudaError_t launch_score(const Dims& d, const void* q_spec, const void* k_dev, float* logits,
                         float2* part, cudaStream_t st) {
  return launch_any<false>(d, q_spec, k_dev, logits, part, FusedOut{}, st);
}

cudaError_t launch_score_bf16_query(const Dims& d, const void* q_bf16, const void* k_f32,
                                    float* logits, float2* part, cudaStream_t st) {
  if (d.dtype != DD_F32) return cudaErrorInvalidValue;
  const FusedOut fo{};
  switch (d.d * 16 + d.G) {
    case 64 * 16 + 1: return launch_typed<float, 64, 1, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 64 * 16 + 2: return launch_typed<float, 64, 2, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 64 * 16 + 4: return launch_typed<float, 64, 4, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 64 * 16 + 8: return launch_typed<float, 64, 8, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 128 * 16 + 1: return launch_typed<float, 128, 1, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 128 * 16 + 2: return launch_typed<float, 128, 2, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 128 * 16 + 4: return launch_typed<float, 128, 4, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
    case 128 * 16 + 8: return launch_typed<float, 128, 8, false, true>(d, q_bf16, k_f32, logits, part, fo, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_score_select(const Dims& d, const void* q_spec, const void* k_dev,
                                float* logits, float2* part, int32_t* counters, int32_t* idx,
                                float* sel, float* lse, cudaStream_t st) {
  const FusedOut fo{counters, idx, sel, lse, d.span, d.k};
  return launch_any<true>(d, q_spec, k_dev, logits, part, fo, st);
}

unsigned int take_score_status() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_score_status, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_score_status, &zero, sizeof zero);
  return v;
}

}  // namespace dd
