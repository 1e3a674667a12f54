/*
 * gen.c - host implementation of the seeded synthetic input generator.
 * Definitions are in gen_core.h; the device twin is gen_cuda.cu.  This file
 * holds no arithmetic of the MoE layer itself.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gen_core.h"

#define GEN_API __attribute__((visibility("default")))

static const double kSd = GEN_IH_SD;

/* activations: row t is draw (draw0 + t) of layer `layer`; bf16 N(0,1) */
GEN_API void gen_x_bf16(uint64_t seed, int layer, int64_t draw0, int T, int H, uint16_t* out) {
  const float c = (float)(1.0 / kSd);
  for (int t = 0; t < T; ++t) {
    uint64_t key = gen_key(seed, GEN_KIND_X, (uint64_t)layer, (uint64_t)(draw0 + t));
    for (int i = 0; i < H; ++i) {
      float v = (float)gen_ih(gen_draw(key, (uint64_t)i)) * c;
      out[(size_t)t * H + i] = gen_f32_to_bf16(v);
    }
  }
}

/* router weights [E][H], fp32 N(0, 0.05^2) */
GEN_API void gen_router_f32(uint64_t seed, int layer, int E, int H, float* out) {
  const float c = (float)(0.05 / kSd);
  for (int e = 0; e < E; ++e) {
    uint64_t key = gen_key(seed, GEN_KIND_ROUTER, (uint64_t)layer, (uint64_t)e);
    for (int i = 0; i < H; ++i)
      out[(size_t)e * H + i] = (float)gen_ih(gen_draw(key, (uint64_t)i)) * c;
  }
}

/* shared expert, bf16 N(0, 0.02^2): gate [Is][H], up [Is][H], down [H][Is] */
GEN_API void gen_shared_bf16(uint64_t seed, int layer, int Is, int H, uint16_t* gate,
                             uint16_t* up, uint16_t* down) {
  const float c = (float)(0.02 / kSd);
  uint16_t* dst[3] = {gate, up, down};
  size_t n = (size_t)Is * (size_t)H;
  for (int m = 0; m < 3; ++m) {
    if (!dst[m]) continue;
    uint64_t key = gen_key(seed, GEN_KIND_SHARED, (uint64_t)layer, (uint64_t)m);
    for (size_t i = 0; i < n; ++i)
      dst[m][i] = gen_f32_to_bf16((float)gen_ih(gen_draw(key, (uint64_t)i)) * c);
  }
}

/* per-(expert, matrix) fp32 global scale g = (0.02 * 64 / sd) * f, with a
 * seeded factor f in [0.875, 1.125) so that experts and matrices differ. */
GEN_API void gen_global_scales(uint64_t seed, int layer, int E, float* g /* [E][3] */) {
  const float base = (float)(0.02 * 64.0 / kSd);
  for (int e = 0; e < E; ++e)
    for (int m = 0; m < 3; ++m) {
      uint64_t h = gen_key(seed, GEN_KIND_GSCALE, (uint64_t)layer, (uint64_t)(e * 4 + m));
      float f = 0.875f + (float)(h >> 56) / 1024.0f;
      g[e * 3 + m] = base * f;
    }
}

/* one matrix (rows [r0, r1)) of one expert record in format fmt */
static void gen_matrix_rows(uint64_t seed, int layer, int expert, int H, int I, int m, int r0,
                            int r1, int fmt, uint8_t* rec) {
  int K = (m == 2) ? I : H;
  int bl = gen_block_len(fmt), KB = K / bl;
  uint64_t key = gen_key(seed, GEN_KIND_EXPERT, (uint64_t)layer, (uint64_t)(expert * 4 + m));
  uint8_t* codes = rec + gen_codes_off(H, I, m);
  uint8_t* scales = rec + gen_scales_off(H, I, m, fmt);
  for (int r = r0; r < r1; ++r)
    for (int kb = 0; kb < KB; ++kb) {
      uint8_t c[16];
      int sb = fmt ? gen_expert_block_mx(key, r, kb, K, c) : gen_expert_block(key, r, kb, K, c);
      memcpy(codes + (size_t)r * (K / 2) + (size_t)kb * (bl / 2), c, (size_t)bl / 2);
      scales[gen_scale_index(r, kb, KB)] = (uint8_t)sb;
    }
}

GEN_API uint64_t gen_record_size(int H, int I, int fmt) { return gen_record_bytes(H, I, fmt); }

GEN_API void gen_expert_record(uint64_t seed, int layer, int expert, int H, int I, int fmt,
                               uint8_t* rec) {
  gen_matrix_rows(seed, layer, expert, H, I, 0, 0, I, fmt, rec);
  gen_matrix_rows(seed, layer, expert, H, I, 1, 0, I, fmt, rec);
  gen_matrix_rows(seed, layer, expert, H, I, 2, 0, H, fmt, rec);
}

/* ---- threaded fill of several records ---- */
typedef struct {
  uint64_t seed;
  int layer, H, I, n, fmt;
  const int32_t* experts;
  uint8_t* const* dst;
  int64_t n_units; /* units = (record, matrix, 64-row chunk) */
  int64_t next;
  pthread_mutex_t mu;
} gen_job;

static void unit_decode(const gen_job* j, int64_t u, int* rec, int* m, int* r0, int* r1) {
  int gu_chunks = (j->I + 63) / 64, d_chunks = (j->H + 63) / 64;
  int per = 2 * gu_chunks + d_chunks;
  *rec = (int)(u / per);
  int w = (int)(u % per);
  if (w < 2 * gu_chunks) {
    *m = w / gu_chunks;
    *r0 = (w % gu_chunks) * 64;
    *r1 = *r0 + 64 < j->I ? *r0 + 64 : j->I;
  } else {
    *m = 2;
    *r0 = (w - 2 * gu_chunks) * 64;
    *r1 = *r0 + 64 < j->H ? *r0 + 64 : j->H;
  }
}

static void* gen_worker(void* arg) {
  gen_job* j = (gen_job*)arg;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int64_t u = j->next;
    j->next += 4;
    pthread_mutex_unlock(&j->mu);
    if (u >= j->n_units) break;
    int64_t ue = u + 4 < j->n_units ? u + 4 : j->n_units;
    for (; u < ue; ++u) {
      int rec, m, r0, r1;
      unit_decode(j, u, &rec, &m, &r0, &r1);
      gen_matrix_rows(j->seed, j->layer, j->experts[rec], j->H, j->I, m, r0, r1, j->fmt,
                      j->dst[rec]);
    }
  }
  return NULL;
}

GEN_API void gen_expert_records_mt(uint64_t seed, int layer, const int32_t* experts, int n, int H,
                                   int I, int fmt, uint8_t* const* dst, int nthreads) {
  gen_job j;
  j.seed = seed; j.layer = layer; j.H = H; j.I = I; j.n = n; j.fmt = fmt;
  j.experts = experts; j.dst = dst; j.next = 0;
  j.n_units = (int64_t)n * (2 * ((I + 63) / 64) + (H + 63) / 64);
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gen_worker, &j);
  gen_worker(&j);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&j.mu);
}

/* ---- per-layer Zipf popularity bias: b_e = -alpha * ln(rank(e)), rank in 1..E,
 * rank = a seeded permutation (Fisher-Yates on draws of the PERM stream). ---- */
GEN_API void gen_zipf_bias(uint64_t seed, int layer, int E, double alpha, float* bias,
                           int32_t* rank_of) {
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int i = 0; i < E; ++i) order[i] = i;
  uint64_t key = gen_key(seed, GEN_KIND_PERM, (uint64_t)layer, 0);
  for (int i = E - 1; i > 0; --i) {
    uint64_t u = gen_draw(key, (uint64_t)i);
    int j = (int)(u % (uint64_t)(i + 1));
    int32_t t = order[i]; order[i] = order[j]; order[j] = t;
  }
  /* order[p] = expert holding popularity position p (rank p + 1) */
  for (int p = 0; p < E; ++p) {
    int e = order[p];
    if (rank_of) rank_of[e] = p + 1;
    if (bias) bias[e] = (float)(-alpha * log((double)(p + 1)));
  }
  free(order);
}

/* pre-quantisation integers d of one row of matrix m of an expert (for the
 * format pins: the represented weight must lie within half a code step of
 * d * g / 64) */
GEN_API void gen_expert_prequant_row(uint64_t seed, int layer, int expert, int H, int I, int m,
                                     int r, int32_t* out) {
  int K = (m == 2) ? I : H;
  uint64_t key = gen_key(seed, GEN_KIND_EXPERT, (uint64_t)layer, (uint64_t)(expert * 4 + m));
  for (int c = 0; c < K; ++c) out[c] = gen_ih(gen_draw(key, (uint64_t)r * (uint64_t)K + (uint64_t)c));
}

GEN_API uint64_t gen_mix64_export(uint64_t z) { return gen_mix64(z); }
