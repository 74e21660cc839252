/*
 * Seeded synthetic workload generator for the predictive sparse-KV decode step.
 *
 * This file holds only input generation: it computes none of the method's
 * arithmetic (no scoring, selection, gather or attention).  Both the fp64
 * oracle and the CUDA path are fed from the buffers it fills.
 *
 * Random numbers come from a counter-based stream built on SplitMix64
 * (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): output i of the stream with base state b is
 * mix(b + (i + 1) * 0x9E3779B97F4A7C15), where mix is the SplitMix64
 * finaliser.  Every element is therefore a pure function of
 * (seed, tensor tag, element index), so any range can be filled by any
 * thread, and a single unit can be regenerated on its own.
 * Normal deviates use the Box-Muller transform (Box & Muller, 1958) on the
 * pair of uniforms (2p, 2p+1).
 *
 * Recipe (per configuration and layer slot), as a workload of the shape of
 * the DualDecoder paper's LLaMA-2-7B/13B long-context decode steps:
 *   q_spec ~ N(0,1); q = q_spec + 0.1 N(0,1);
 *   K, V ~ N(0,1) (optionally K row j scaled by s_j ~ LogNormal(0, 0.5),
 *   one scale per (request, token) shared by all heads);
 *   P planted keys per KV head: K_i = 3 sqrt(d) u + 0.1 N(0,1), with u the
 *   unit direction of q_spec (MHA) or the normalised sum of the group's
 *   unit q_spec directions (GQA).
 * Values are generated in fp32 and rounded to nearest-even bf16 when the
 * stored dtype is bf16.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

enum { SYN_F32 = 0, SYN_BF16 = 1 };
enum {
  TAG_QSPEC = 1,
  TAG_QNOISE = 2,
  TAG_K = 3,
  TAG_V = 4,
  TAG_PLANT_POS = 5,
  TAG_PLANT_NOISE = 6,
  TAG_KSCALE = 7
};
enum { PLANT_NONE = 0, PLANT_RANDOM = 1, PLANT_SPREAD = 2 };

static inline uint64_t syn_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Base state of the stream for (seed, tag). */
uint64_t syn_stream(uint64_t seed, uint64_t tag) {
  return syn_mix(syn_mix(seed) ^ (tag * SYN_GAMMA));
}

/* i-th 64-bit output of a stream. */
uint64_t syn_u64(uint64_t base, uint64_t i) {
  return syn_mix(base + (i + 1) * SYN_GAMMA);
}

/* Uniform in the open interval (0, 1), 53 bits. */
static inline double syn_unif(uint64_t base, uint64_t i) {
  return ((double)(syn_u64(base, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* e-th standard normal of a stream (Box-Muller over the uniform pair). */
double syn_normal(uint64_t base, uint64_t e) {
  uint64_t p = e >> 1;
  double u1 = syn_unif(base, 2 * p);
  double u2 = syn_unif(base, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (e & 1) ? r * sin(th) : r * cos(th);
}

/* Both normals of pair p: elements 2p (cosine) and 2p+1 (sine). */
static inline void syn_normal_pair(uint64_t base, uint64_t p, double* z0, double* z1) {
  double u1 = syn_unif(base, 2 * p);
  double u2 = syn_unif(base, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(th);
  *z1 = r * sin(th);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

static inline void store(void* buf, int dtype, int64_t i, float v) {
  if (dtype == SYN_BF16)
    ((uint16_t*)buf)[i] = f32_to_bf16_rne(v);
  else
    ((float*)buf)[i] = v;
}

typedef struct {
  int32_t batch, n_q_heads, n_kv_heads, head_dim, ctx_len, window;
  int32_t dtype;      /* SYN_F32 or SYN_BF16 */
  int32_t n_planted;  /* planted keys per KV head */
  int32_t plant_mode; /* PLANT_NONE / PLANT_RANDOM / PLANT_SPREAD */
  int32_t key_scale;  /* 1: per-(request, token) LogNormal(0, 0.5) key scale */
  float q_noise;      /* standard deviation of q - q_spec */
  float plant_noise;  /* standard deviation of the planted-key noise */
  float plant_gain;   /* planted key = plant_gain * sqrt(d) * u + noise */
} syn_cfg;

/* ---- small thread pool: split [0, count) into nthreads contiguous ranges ---- */
typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct {
  range_fn fn;
  void* ctx;
  int64_t lo, hi;
} range_job;

static void* range_tramp(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t count, int nthreads, range_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (count < (int64_t)nthreads * 4096) nthreads = 1;
  if (nthreads == 1) {
    fn(ctx, 0, count);
    return;
  }
  pthread_t th[256];
  int live[256];
  range_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].lo = count * t / nthreads;
    jobs[t].hi = count * (t + 1) / nthreads;
    live[t] = pthread_create(&th[t], NULL, range_tramp, &jobs[t]) == 0;
    if (!live[t]) range_tramp(&jobs[t]); /* no thread: run the range inline */
  }
  for (int t = 0; t < nthreads; ++t)
    if (live[t]) pthread_join(th[t], NULL);
}

/* ---- plain normal fill: out[i] = mean + sd * N(offset + i) ---- */
typedef struct {
  uint64_t base, offset;
  void* out;
  int dtype;
  float mean, sd;
} fill_ctx;

static void fill_range(void* p, int64_t lo, int64_t hi) {
  fill_ctx* c = (fill_ctx*)p;
  int64_t i = lo;
  /* whole pairs of the stream where possible, single elements at the ends */
  while (i < hi && ((c->offset + (uint64_t)i) & 1)) {
    store(c->out, c->dtype, i, c->mean + c->sd * (float)syn_normal(c->base, c->offset + (uint64_t)i));
    ++i;
  }
  for (; i + 1 < hi; i += 2) {
    double z0, z1;
    syn_normal_pair(c->base, (c->offset + (uint64_t)i) >> 1, &z0, &z1);
    store(c->out, c->dtype, i, c->mean + c->sd * (float)z0);
    store(c->out, c->dtype, i + 1, c->mean + c->sd * (float)z1);
  }
  if (i < hi)
    store(c->out, c->dtype, i, c->mean + c->sd * (float)syn_normal(c->base, c->offset + (uint64_t)i));
}

void syn_fill_normal(uint64_t seed, uint64_t tag, uint64_t offset, int64_t count,
                     float mean, float sd, int dtype, void* out, int nthreads) {
  fill_ctx c = {syn_stream(seed, tag), offset, out, dtype, mean, sd};
  parallel_for(count, nthreads, fill_range, &c);
}

/* ---- queries ----
 * q_spec[b][h][t] = N_QSPEC(e), q = q_spec + q_noise * N_QNOISE(e),
 * with e = (b*H_q + h)*d + t.  Both are rounded from the fp32 values.
 * qspec_f32 (optional, may be NULL) receives the unrounded q_spec.         */
void syn_queries(const syn_cfg* c, uint64_t seed, void* q_spec, void* q, float* qspec_f32) {
  int64_t count = (int64_t)c->batch * c->n_q_heads * c->head_dim;
  uint64_t bs = syn_stream(seed, TAG_QSPEC), bn = syn_stream(seed, TAG_QNOISE);
  for (int64_t e = 0; e < count; ++e) {
    float qs = (float)syn_normal(bs, (uint64_t)e);
    float qq = qs + c->q_noise * (float)syn_normal(bn, (uint64_t)e);
    if (qspec_f32) qspec_f32[e] = qs;
    store(q_spec, c->dtype, e, qs);
    store(q, c->dtype, e, qq);
  }
}

/* ---- planted positions for one KV head unit u = b*H_kv + h ----
 * PLANT_RANDOM: P distinct positions, uniform in [0, n - W), drawn in order
 *   from the TAG_PLANT_POS stream at counters u*2^32 + draw (rejection of
 *   repeats).  PLANT_SPREAD: floor((i + 1/2)(n - W)/P).                    */
void syn_planted_positions(const syn_cfg* c, uint64_t seed, int64_t unit, int32_t* pos) {
  int32_t P = c->n_planted, span = c->ctx_len - c->window;
  if (P <= 0 || c->plant_mode == PLANT_NONE) return;
  if (c->plant_mode == PLANT_SPREAD) {
    for (int i = 0; i < P; ++i)
      pos[i] = (int32_t)(((int64_t)(2 * i + 1) * span) / (2 * (int64_t)P));
    return;
  }
  uint64_t base = syn_stream(seed, TAG_PLANT_POS);
  uint64_t draw = 0;
  for (int i = 0; i < P; ++i) {
    for (;;) {
      uint64_t x = syn_u64(base, ((uint64_t)unit << 32) + draw++);
      int32_t cand = (int32_t)(((x >> 11) * (uint64_t)span) >> 53);
      int dup = 0;
      for (int r = 0; r < i; ++r) dup |= (pos[r] == cand);
      if (!dup) {
        pos[i] = cand;
        break;
      }
    }
  }
}

/* ---- K and V ---- */
typedef struct {
  const syn_cfg* c;
  uint64_t bk, bv, bscale;
  void *K, *V;
} kv_ctx;

/* Range over rows r = (b*H_kv + h)*n + j. */
static void kv_range(void* p, int64_t lo, int64_t hi) {
  kv_ctx* x = (kv_ctx*)p;
  const syn_cfg* c = x->c;
  int64_t d = c->head_dim, n = c->ctx_len;
  for (int64_t r = lo; r < hi; ++r) {
    float scale = 1.0f;
    if (c->key_scale) {
      int64_t j = r % n, b = (r / n) / c->n_kv_heads;
      scale = (float)exp(0.5 * syn_normal(x->bscale, (uint64_t)(b * n + j)));
    }
    /* d is even, so the row's elements are whole pairs of the stream */
    for (int64_t t = 0; t < d; t += 2) {
      uint64_t pr = (uint64_t)(r * d + t) >> 1;
      double z0, z1;
      if (x->K) {
        syn_normal_pair(x->bk, pr, &z0, &z1);
        store(x->K, c->dtype, r * d + t, scale * (float)z0);
        store(x->K, c->dtype, r * d + t + 1, scale * (float)z1);
      }
      if (x->V) {
        syn_normal_pair(x->bv, pr, &z0, &z1);
        store(x->V, c->dtype, r * d + t, (float)z0);
        store(x->V, c->dtype, r * d + t + 1, (float)z1);
      }
    }
  }
}

/* Direction used by planted keys of unit (b, h_kv): the unit q_spec of the
 * head (MHA) or the normalised sum of the group's unit q_spec directions.   */
static void planted_direction(const syn_cfg* c, const float* qspec_f32, int b, int hk, double* u) {
  int d = c->head_dim, G = c->n_q_heads / c->n_kv_heads;
  for (int t = 0; t < d; ++t) u[t] = 0.0;
  for (int g = 0; g < G; ++g) {
    const float* qs = qspec_f32 + ((int64_t)b * c->n_q_heads + (int64_t)hk * G + g) * d;
    double nrm = 0.0;
    for (int t = 0; t < d; ++t) nrm += (double)qs[t] * qs[t];
    nrm = sqrt(nrm);
    for (int t = 0; t < d; ++t) u[t] += qs[t] / nrm;
  }
  double nrm = 0.0;
  for (int t = 0; t < d; ++t) nrm += u[t] * u[t];
  nrm = sqrt(nrm);
  for (int t = 0; t < d; ++t) u[t] /= nrm;
}

/*
 * Fill K and V ([B][H_kv][n][d]) for one layer slot and overwrite the
 * planted rows.  qspec_f32 is the unrounded q_spec from syn_queries.
 * planted (optional) receives [B][H_kv][P] positions.  K or V may be NULL.
 */
void syn_kv(const syn_cfg* c, uint64_t seed, const float* qspec_f32, void* K, void* V,
            int32_t* planted, int nthreads) {
  kv_ctx x = {c, syn_stream(seed, TAG_K), syn_stream(seed, TAG_V), syn_stream(seed, TAG_KSCALE),
              K, V};
  int64_t rows = (int64_t)c->batch * c->n_kv_heads * c->ctx_len;
  parallel_for(rows, nthreads, kv_range, &x);
  if (c->n_planted <= 0 || c->plant_mode == PLANT_NONE) return;
  int d = c->head_dim, P = c->n_planted;
  double* u = (double*)malloc(sizeof(double) * d);
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * P);
  uint64_t bn = syn_stream(seed, TAG_PLANT_NOISE);
  double gain = c->plant_gain * sqrt((double)d);
  for (int b = 0; b < c->batch; ++b)
    for (int hk = 0; hk < c->n_kv_heads; ++hk) {
      int64_t unit = (int64_t)b * c->n_kv_heads + hk;
      syn_planted_positions(c, seed, unit, pos);
      if (planted) memcpy(planted + unit * P, pos, sizeof(int32_t) * P);
      planted_direction(c, qspec_f32, b, hk, u);
      for (int i = 0; i < P; ++i) {
        int64_t row = unit * c->ctx_len + pos[i];
        for (int t = 0; t < d; ++t) {
          float v = (float)(gain * u[t]) +
                    c->plant_noise * (float)syn_normal(bn, (uint64_t)((unit * P + i) * d + t));
          if (K) store(K, c->dtype, row * d + t, v);
        }
      }
    }
  free(u);
  free(pos);
}
