/* Host fills of the seeded synthetic-input generator (definition in
 * dsgen_core.h).  Test and benchmark infrastructure: serves both the oracle
 * and the CUDA path, holds none of the MoE method's arithmetic. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include "dsgen_core.h"

float dsgen_scale_normal(double sigma) { return (float)(sigma * sqrt(12.0 / 8.0) / 65536.0); }
float dsgen_scale_uniform(double a) { return (float)(a / 16777216.0); }

typedef struct {
  float *out; uint16_t *out_bf16; uint64_t lo, hi, idx0;
  uint32_t seed, layer, tensor, sub; float c; int uniform;
} fill_job;

static void *fill_worker(void *p) {
  fill_job *j = (fill_job *)p;
  for (uint64_t i = j->lo; i < j->hi; ++i) {
    float v = j->uniform ? dsgen_uniform(j->seed, j->layer, j->tensor, j->sub, j->idx0 + i, j->c)
                         : dsgen_normal(j->seed, j->layer, j->tensor, j->sub, j->idx0 + i, j->c);
    if (j->out) j->out[i] = v;
    if (j->out_bf16) j->out_bf16[i] = dsgen_f32_to_bf16(v);
  }
  return NULL;
}

static void fill(float *out, uint16_t *out_bf16, uint64_t n, uint32_t seed, uint32_t layer,
                 uint32_t tensor, uint32_t sub, uint64_t idx0, float c, int uniform, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 65536) nthreads = 1;
  pthread_t th[256];
  fill_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    fill_job j = {out, out_bf16, n * (uint64_t)t / (uint64_t)nthreads,
                  n * (uint64_t)(t + 1) / (uint64_t)nthreads, idx0, seed, layer, tensor, sub, c, uniform};
    jobs[t] = j;
  }
  if (nthreads == 1) { fill_worker(&jobs[0]); return; }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* out[i] = normal(idx0 + i), i < n; out_bf16 (optional) = its bf16 rounding. */
void dsgen_fill_normal(float *out, uint16_t *out_bf16, uint64_t n, uint32_t seed, uint32_t layer,
                       uint32_t tensor, uint32_t sub, uint64_t idx0, float c, int nthreads) {
  fill(out, out_bf16, n, seed, layer, tensor, sub, idx0, c, 0, nthreads);
}

void dsgen_fill_uniform(float *out, uint16_t *out_bf16, uint64_t n, uint32_t seed, uint32_t layer,
                        uint32_t tensor, uint32_t sub, uint64_t idx0, float c, int nthreads) {
  fill(out, out_bf16, n, seed, layer, tensor, sub, idx0, c, 1, nthreads);
}

/* Activation rows: row t is drawn with sub = attempt[t] (resample counter),
 * idx = t*D + d.  attempt may be NULL (all zero). */
void dsgen_x_rows(float *out, uint16_t *out_bf16, int64_t T, int64_t D, const int32_t *attempt,
                  uint32_t seed, uint32_t layer, float c) {
  for (int64_t t = 0; t < T; ++t) {
    uint32_t a = attempt ? (uint32_t)attempt[t] : 0u;
    for (int64_t d = 0; d < D; ++d) {
      float v = dsgen_normal(seed, layer, DSGEN_T_X, a, (uint64_t)(t * D + d), c);
      if (out) out[t * D + d] = v;
      if (out_bf16) out_bf16[t * D + d] = dsgen_f32_to_bf16(v);
    }
  }
}

/* Seeded Fisher-Yates shuffle of the ranks 1..E; rank[e] is expert e's
 * popularity rank.  Draw i uses idx = i of tensor DSGEN_T_ZIPF_PERM. */
void dsgen_zipf_ranks(int32_t *rank, int32_t E, uint32_t seed, uint32_t layer) {
  for (int32_t e = 0; e < E; ++e) rank[e] = e + 1;
  for (int32_t i = E - 1; i > 0; --i) {
    uint32_t r[4];
    dsgen_draw(seed, layer, DSGEN_T_ZIPF_PERM, 0, (uint64_t)i, r);
    int32_t j = (int32_t)(r[0] % (uint32_t)(i + 1));
    int32_t tmp = rank[i]; rank[i] = rank[j]; rank[j] = tmp;
  }
}

void dsgen_to_bf16(const float *in, uint16_t *out, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) out[i] = dsgen_f32_to_bf16(in[i]);
}

void dsgen_philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1,
                  uint32_t *out4) {
  dsgen_philox4x32_10(c0, c1, c2, c3, k0, k1, out4);
}
