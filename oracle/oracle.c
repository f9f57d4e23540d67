/* Oracle for the routed mixture-of-experts layer with 2-bit (Q2_K) experts.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, fp64 CPU code that defines what the
 * layer computes.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path never does.  It shares no code with
 * the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [UDS]  "Understanding Dwarf Star" (ldazrz.com):
 *          3.3.3 "Q2_K: 2.625 Bits Per Element" (84-byte block of 256
 *          weights, fp16 super-block scale and min, 16 sub-blocks of 16);
 *          2.3.5 (the 4 levels are evenly spaced between min and max);
 *          2.8.1 (weights are reconstructed from stored scales and mins);
 *          5.3.2 "The MoE Architecture" (router(x) = softmax(x W_router),
 *          top-k selection, weighted sum of expert outputs, 256 experts,
 *          top-6, one always-active shared expert);
 *          5.2.4 (SwiGLU / SiLU feed-forward network);
 *          5.3.7 "The MoE Kernel in Metal" (gate projection -> activation ->
 *          down projection, multiply by router weight and accumulate);
 *          2.4.3 (shape table: n_embd 4096, 43 layers, 256 experts, 6 used,
 *          1 shared, n_ff_exp 2048).
 *   [YD]   "The sparsity that pays for everything else in DwarfStar"
 *          (yashdatta.dev), "Where the parameters actually are" (gate, up
 *          and down per expert; 3 x 4096 x 2048 parameters per expert).
 *
 * Readings where the pages are silent:
 *   - Block byte layout: bytes [0,16) hold sub-block s's scale (low nibble)
 *     and min (high nibble); [16,80) the 2-bit codes, weight j at byte
 *     16 + j/4, bits 2*(j%4); [80,82) d and [82,84) dmin, fp16 little-endian.
 *     w_j = d*sc_s*q_j - dmin*m_s.
 *   - Quantiser: per sub-block lo_s = min(0, min x), hi_s = max x;
 *     dmin = smallest fp16 >= max_s(-lo_s)/15; m_s = smallest integer with
 *     m_s*dmin >= -lo_s; b_s = dmin*m_s; d = smallest fp16 >= max_s(hi_s+b_s)/45;
 *     sc_s = smallest integer with 3*d*sc_s >= hi_s + b_s;
 *     q_j = clamp(floor((x_j + b_s)/(d*sc_s) + 1/2), 0, 3) (0 when sc_s = 0).
 *     Every quantity is evaluated exactly (the comparisons below are exact
 *     in fp64), so the result is the formula's value, not a rounding of it.
 *   - Rows whose length is not a multiple of 256 are zero-padded.
 *   - Routing: logits in fp64 (the kernel's fp32), top-k by logit with ties
 *     to the lower expert index, weights = softmax over the selected logits
 *     (equal to the full softmax renormalised over the k selected), times
 *     routed_scale (1 by default).
 *   - The shared expert is added unweighted; output is summed as
 *     y_shared + sum_j w_j y_j in slot order j.
 *   - Stack: x <- fp32(x + layer(bf16(x / sqrt(mean(x^2) + 1e-6)))).
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against
 * values the pages print, closed forms, brute force or special cases.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 256
#define QBYTES 84

/* ---------------------------------------------------------------- fp16 --- */

/* Value of an IEEE binary16 bit pattern. */
double oracle_fp16_value(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m + 1024), e - 25);
  return s ? -v : v;
}

/* Smallest non-negative finite fp16 h with ok(h) true, where ok is monotone
 * in h.  Non-negative fp16 values are ordered like their bit patterns, so a
 * binary search over 0x0000..0x7BFF finds it.  Returns -1 if none. */
typedef int (*fp16_pred)(double h, const void *ctx);
static int fp16_smallest(fp16_pred ok, const void *ctx) {
  int lo = 0, hi = 0x7BFF;
  if (!ok(oracle_fp16_value((uint16_t)hi), ctx)) return -1;
  while (lo < hi) {
    int mid = (lo + hi) / 2;
    if (ok(oracle_fp16_value((uint16_t)mid), ctx)) hi = mid; else lo = mid + 1;
  }
  return lo;
}

typedef struct { const double *neg_lo; } dmin_ctx;
/* 15*h >= max_s(-lo_s); 15*h is exact in fp64. */
static int dmin_ok(double h, const void *c) {
  const dmin_ctx *x = (const dmin_ctx *)c;
  for (int s = 0; s < 16; ++s) if (15.0 * h < x->neg_lo[s]) return 0;
  return 1;
}

typedef struct { const double *hi, *b; } d_ctx;
/* 45*h >= hi_s + b_s for all s, tested as 45*h - b_s >= hi_s: 45*h - b_s is
 * exact in fp64 (both operands are fp16 values times integers below 64, so
 * the difference spans at most 47 bits). */
static int d_ok(double h, const void *c) {
  const d_ctx *x = (const d_ctx *)c;
  for (int s = 0; s < 16; ++s) if (45.0 * h - x->b[s] < x->hi[s]) return 0;
  return 1;
}

/* ----------------------------------------------------------- Q2_K block --- */

/* Quantise one super-block of 256 values ([UDS] 3.3.3, reading above).
 * Returns 0, or -1 when a value is not finite or |v| > 65504 (the largest
 * fp16: the encoding's domain, so that every scale fits in fp16). */
static int q2k_quantize_block(const double *x, uint8_t *out) {
  double lo[16], hi[16], neg_lo[16], b[16];
  int m[16], sc[16];
  for (int s = 0; s < 16; ++s) {
    double mn = 0.0, mx = -INFINITY;
    for (int j = 0; j < 16; ++j) {
      double v = x[16 * s + j];
      if (!(fabs(v) <= 65504.0)) return -1; /* also rejects NaN and infinities */
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    lo[s] = mn;
    hi[s] = mx;
    neg_lo[s] = -mn;
  }
  dmin_ctx dc = {neg_lo};
  int dmin_bits = fp16_smallest(dmin_ok, &dc);
  if (dmin_bits < 0) return -1;
  double dmin = oracle_fp16_value((uint16_t)dmin_bits);
  for (int s = 0; s < 16; ++s) {
    int mm = 0;
    while (mm < 15 && (double)mm * dmin < -lo[s]) ++mm;
    m[s] = mm;
    b[s] = (double)mm * dmin; /* exact */
  }
  d_ctx cx = {hi, b};
  int d_bits = fp16_smallest(d_ok, &cx);
  if (d_bits < 0) return -1;
  double d = oracle_fp16_value((uint16_t)d_bits);
  for (int s = 0; s < 16; ++s) {
    int c = 0;
    while (c < 15 && 3.0 * d * (double)c - b[s] < hi[s]) ++c; /* exact */
    sc[s] = c;
  }
  memset(out, 0, QBYTES);
  for (int s = 0; s < 16; ++s) out[s] = (uint8_t)(sc[s] | (m[s] << 4));
  for (int j = 0; j < QK; ++j) {
    int s = j / 16, q = 0;
    if (sc[s] > 0) {
      for (int i = 1; i <= 3; ++i) {
        /* (i - 1/2)*d*sc - b is exact in fp64, so is the comparison */
        double thr = ((double)i - 0.5) * d * (double)sc[s] - b[s];
        if (x[j] >= thr) ++q;
      }
    }
    out[16 + j / 4] |= (uint8_t)(q << (2 * (j % 4)));
  }
  out[80] = (uint8_t)(d_bits & 0xFF);
  out[81] = (uint8_t)(d_bits >> 8);
  out[82] = (uint8_t)(dmin_bits & 0xFF);
  out[83] = (uint8_t)(dmin_bits >> 8);
  return 0;
}

/* Dequantise one block: w_j = d*sc_s*q_j - dmin*m_s, exact in fp64
 * ([UDS] 2.8.1: reconstruct from the stored scales and mins). */
static void q2k_dequantize_block(const uint8_t *blk, double *w) {
  double d = oracle_fp16_value((uint16_t)(blk[80] | (blk[81] << 8)));
  double dmin = oracle_fp16_value((uint16_t)(blk[82] | (blk[83] << 8)));
  for (int j = 0; j < QK; ++j) {
    int s = j / 16;
    int sc = blk[s] & 15, m = blk[s] >> 4;
    int q = (blk[16 + j / 4] >> (2 * (j % 4))) & 3;
    w[j] = d * (double)sc * (double)q - dmin * (double)m;
  }
}

/* ----------------------------------------------------------- Q4_K block --- */
/* [UDS] 2.3.2 "K-Quant Formats (Q2_K, Q3_K, Q4_K, etc.)": a 144-byte block of
 * 256 values (4.5 bits per value): an fp16 super-block scale d at offset 0,
 * an fp16 minimum dmin at offset 2, eight 6-bit scales and eight 6-bit mins
 * packed into the 12 bytes at offset 4, and the 256 4-bit values in the 128
 * bytes at offset 16; eight sub-blocks of 32 values.
 * Readings (the page gives the fields, not their packing or the search):
 *   - the sixteen 6-bit fields sc_0..sc_7, m_0..m_7 form one 96-bit
 *     little-endian integer in bytes 4..15, field i in bits [6i, 6i + 6);
 *   - the code of value j sits in byte 16 + j/2, low nibble for even j;
 *   - the quantiser follows the Q2_K rules with 16 levels and 6-bit fields:
 *     dmin = smallest fp16 with 63 dmin >= max_s(-lo_s); m_s = smallest
 *     integer with m_s dmin >= -lo_s; b_s = m_s dmin; d = smallest fp16 with
 *     945 d >= hi_s + b_s for every s; sc_s = smallest integer with
 *     15 d sc_s >= hi_s + b_s; q_j = clamp(floor((x_j + b_s)/(d sc_s) + 1/2),
 *     0, 15) (0 when sc_s = 0); w_j = d sc_s q_j - dmin m_s.  All exact. */
#define Q4BYTES 144
#define Q4SUB 8

static int q4k_get6(const uint8_t *blk, int i) {
  int v = 0;
  for (int k = 0; k < 6; ++k) {
    const int bit = 6 * i + k;
    v |= ((blk[4 + bit / 8] >> (bit % 8)) & 1) << k;
  }
  return v;
}

static void q4k_put6(uint8_t *blk, int i, int v) {
  for (int k = 0; k < 6; ++k) {
    const int bit = 6 * i + k;
    blk[4 + bit / 8] |= (uint8_t)(((v >> k) & 1) << (bit % 8));
  }
}

/* 63*h >= max_s(-lo_s) over the 8 sub-blocks; 63*h is exact in fp64. */
static int q4_dmin_ok(double h, const void *c) {
  const dmin_ctx *x = (const dmin_ctx *)c;
  for (int s = 0; s < Q4SUB; ++s) if (63.0 * h < x->neg_lo[s]) return 0;
  return 1;
}

/* 945*h - b_s >= hi_s for every sub-block; exact in fp64 (fp16 values times
 * integers below 1024, so each side spans well under 53 bits). */
static int q4_d_ok(double h, const void *c) {
  const d_ctx *x = (const d_ctx *)c;
  for (int s = 0; s < Q4SUB; ++s) if (945.0 * h - x->b[s] < x->hi[s]) return 0;
  return 1;
}

/* Quantise one super-block of 256 values (reading above).  Returns 0, or -1
 * when a value is not finite or |v| > 65504. */
static int q4k_quantize_block(const double *x, uint8_t *out) {
  double lo[Q4SUB], hi[Q4SUB], neg_lo[Q4SUB], b[Q4SUB];
  int m[Q4SUB], sc[Q4SUB];
  for (int s = 0; s < Q4SUB; ++s) {
    double mn = 0.0, mx = -INFINITY;
    for (int j = 0; j < 32; ++j) {
      double v = x[32 * s + j];
      if (!(fabs(v) <= 65504.0)) return -1;
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    lo[s] = mn;
    hi[s] = mx;
    neg_lo[s] = -mn;
  }
  dmin_ctx dc = {neg_lo};
  int dmin_bits = fp16_smallest(q4_dmin_ok, &dc);
  if (dmin_bits < 0) return -1;
  double dmin = oracle_fp16_value((uint16_t)dmin_bits);
  for (int s = 0; s < Q4SUB; ++s) {
    int mm = 0;
    while (mm < 63 && (double)mm * dmin < -lo[s]) ++mm;
    m[s] = mm;
    b[s] = (double)mm * dmin; /* exact */
  }
  d_ctx cx = {hi, b};
  int d_bits = fp16_smallest(q4_d_ok, &cx);
  if (d_bits < 0) return -1;
  double d = oracle_fp16_value((uint16_t)d_bits);
  for (int s = 0; s < Q4SUB; ++s) {
    int c = 0;
    while (c < 63 && 15.0 * d * (double)c - b[s] < hi[s]) ++c; /* exact */
    sc[s] = c;
  }
  memset(out, 0, Q4BYTES);
  out[0] = (uint8_t)(d_bits & 0xFF);
  out[1] = (uint8_t)(d_bits >> 8);
  out[2] = (uint8_t)(dmin_bits & 0xFF);
  out[3] = (uint8_t)(dmin_bits >> 8);
  for (int s = 0; s < Q4SUB; ++s) {
    q4k_put6(out, s, sc[s]);
    q4k_put6(out, Q4SUB + s, m[s]);
  }
  for (int j = 0; j < QK; ++j) {
    int s = j / 32, q = 0;
    if (sc[s] > 0)
      for (int i = 1; i <= 15; ++i) {
        double thr = ((double)i - 0.5) * d * (double)sc[s] - b[s]; /* exact */
        if (x[j] >= thr) ++q;
      }
    out[16 + j / 2] |= (uint8_t)(q << (4 * (j % 2)));
  }
  return 0;
}

/* w_j = d*sc_s*q_j - dmin*m_s, exact in fp64. */
static void q4k_dequantize_block(const uint8_t *blk, double *w) {
  double d = oracle_fp16_value((uint16_t)(blk[0] | (blk[1] << 8)));
  double dmin = oracle_fp16_value((uint16_t)(blk[2] | (blk[3] << 8)));
  for (int j = 0; j < QK; ++j) {
    int s = j / 32;
    int q = (blk[16 + j / 2] >> (4 * (j % 2))) & 15;
    w[j] = d * (double)q4k_get6(blk, s) * (double)q - dmin * (double)q4k_get6(blk, Q4SUB + s);
  }
}

int64_t oracle_q2k_blocks_per_row(int64_t in_dim) { return (in_dim + QK - 1) / QK; }
int64_t oracle_q2k_bytes(int64_t rows, int64_t in_dim) {
  return rows * oracle_q2k_blocks_per_row(in_dim) * QBYTES;
}

typedef struct {
  const float *w; int64_t r0, r1, in_dim; uint8_t *out; int err; int q4;
} qjob;

static void *quant_worker(void *p) {
  qjob *j = (qjob *)p;
  int64_t nb = oracle_q2k_blocks_per_row(j->in_dim);
  const int64_t bb = j->q4 ? Q4BYTES : QBYTES;
  double buf[QK];
  for (int64_t r = j->r0; r < j->r1; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      for (int i = 0; i < QK; ++i) {
        int64_t c = b * QK + i;
        buf[i] = c < j->in_dim ? (double)j->w[r * j->in_dim + c] : 0.0; /* zero pad */
      }
      uint8_t *o = j->out + (r * nb + b) * bb;
      if (j->q4 ? q4k_quantize_block(buf, o) : q2k_quantize_block(buf, o)) j->err = 1;
    }
  }
  return NULL;
}

static int quantize_rows(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, int nthreads, int q4) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (rows < nthreads) nthreads = rows > 0 ? (int)rows : 1;
  pthread_t th[256];
  qjob jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    qjob j = {w, rows * t / nthreads, rows * (t + 1) / nthreads, in_dim, out, 0, q4};
    jobs[t] = j;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, quant_worker, &jobs[t]);
  quant_worker(&jobs[0]);
  int err = jobs[0].err;
  for (int t = 1; t < nthreads; ++t) { pthread_join(th[t], NULL); err |= jobs[t].err; }
  return err ? -1 : 0;
}

/* Quantise a row-major fp32 matrix [rows][in_dim] along its rows.
 * out: rows * ceil(in_dim/256) * 84 bytes.  Returns 0 or -1. */
int oracle_q2k_quantize(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, int nthreads) {
  return quantize_rows(w, rows, in_dim, out, nthreads, 0);
}

/* The same with Q4_K blocks: rows * ceil(in_dim/256) * 144 bytes. */
int oracle_q4k_quantize(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, int nthreads) {
  return quantize_rows(w, rows, in_dim, out, nthreads, 1);
}

int64_t oracle_q4k_bytes(int64_t rows, int64_t in_dim) {
  return rows * oracle_q2k_blocks_per_row(in_dim) * Q4BYTES;
}

/* Dequantise Q4_K rows [rows][in_dim] (padding dropped) into fp64. */
void oracle_q4k_dequantize(const uint8_t *q, int64_t rows, int64_t in_dim, double *out) {
  int64_t nb = oracle_q2k_blocks_per_row(in_dim);
  double buf[QK];
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      q4k_dequantize_block(q + (r * nb + b) * Q4BYTES, buf);
      for (int i = 0; i < QK; ++i) {
        int64_t c = b * QK + i;
        if (c < in_dim) out[r * in_dim + c] = buf[i];
      }
    }
}

/* Dequantise [rows][in_dim] (padding dropped) into fp64. */
void oracle_q2k_dequantize(const uint8_t *q, int64_t rows, int64_t in_dim, double *out) {
  int64_t nb = oracle_q2k_blocks_per_row(in_dim);
  double buf[QK];
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      q2k_dequantize_block(q + (r * nb + b) * QBYTES, buf);
      for (int i = 0; i < QK; ++i) {
        int64_t c = b * QK + i;
        if (c < in_dim) out[r * in_dim + c] = buf[i];
      }
    }
}

/* -------------------------------------------------------------- routing --- */

/* logits[t][e] = sum_d x[t][d]*Wr[e][d] (+ bias[e])  ([UDS] 5.3.2:
 * router(x) = softmax(x W_router); Wr is stored [E][D]). */
void oracle_router_logits(const double *x, int64_t T, int64_t D, const double *wr, int64_t E,
                          const double *bias, double *logits) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += x[t * D + d] * wr[e * D + d];
      logits[t * E + e] = acc + (bias ? bias[e] : 0.0);
    }
}

/* Top-k selection and weights for each token ([UDS] 5.3.2: the top-k experts
 * by router probability, weighted by the router probabilities).  Selection
 * by logit, ties to the lower index, in descending order; the weights are the
 * softmax over logit_scale times the k selected logits ([UDS] 5.3.5: a scale
 * applied "before softmax"; 1 = plain softmax), times routed_scale ([UDS]
 * 5.3.2: "a multiplier on router probabilities").  unbias (or null): the
 * router bias, taken back out of the selected logits for the weights when it
 * is to steer the selection only. */
void oracle_select(const double *logits, int64_t T, int64_t E, int32_t k, double routed_scale,
                   double logit_scale, const double *unbias, int32_t *ids, double *w) {
  char *taken = (char *)malloc((size_t)E);
  double *u = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  for (int64_t t = 0; t < T; ++t) {
    const double *L = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int32_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || L[e] > L[best])) best = e; /* strict: lower index wins ties */
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
    }
    /* the weights' logits: with unbias (the router bias, when it steers the
     * selection only) the bias is taken back out of the selected logits */
    double mx = 0.0, den = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      const int32_t e = ids[t * k + j];
      u[j] = L[e] - (unbias ? unbias[e] : 0.0);
      if (j == 0 || u[j] > mx) mx = u[j];
    }
    for (int32_t j = 0; j < k; ++j) den += exp(logit_scale * (u[j] - mx));
    for (int32_t j = 0; j < k; ++j) w[t * k + j] = routed_scale * exp(logit_scale * (u[j] - mx)) / den;
  }
  free(u);
  free(taken);
}

/* Expert histogram, exclusive scan and stable token permutation:
 * counts[e] = #{(t,j): ids[t][j] = e}; offsets = exclusive scan (E+1 entries);
 * perm[offsets[e] + r] = t*k + j for the r-th such pair in ascending t*k+j;
 * pos[t*k + j] = its position in perm. */
void oracle_route(const int32_t *ids, int64_t T, int32_t k, int64_t E, int32_t *counts,
                  int32_t *offsets, int32_t *perm, int32_t *pos) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < T * k; ++p) counts[ids[p]]++;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  for (int64_t p = 0; p < T * k; ++p) {
    int32_t e = ids[p];
    int32_t at = offsets[e] + fill[e]++;
    perm[at] = (int32_t)p;
    if (pos) pos[p] = at;
  }
  free(fill);
}

/* ------------------------------------------------------------ expert FFN --- */

static double silu(double z) { return z / (1.0 + exp(-z)); } /* [UDS] 5.2.4 */

/* Expert storage formats: 0 = Q2_K (84-byte blocks), 1 = Q4_K (144-byte
 * blocks).  Both store a matrix row by row along its input dimension. */
static int64_t fmt_bytes(int fmt, int64_t rows, int64_t in_dim) {
  return fmt ? oracle_q4k_bytes(rows, in_dim) : oracle_q2k_bytes(rows, in_dim);
}

static void fmt_dequantize(int fmt, const uint8_t *q, int64_t rows, int64_t in_dim, double *out) {
  if (fmt) oracle_q4k_dequantize(q, rows, in_dim, out);
  else oracle_q2k_dequantize(q, rows, in_dim, out);
}

/* Bytes of one routed expert: gate [F][D], up [F][D], down [D][F], each
 * in the expert format along its input dimension ([YD]: gate, up and down
 * per expert). */
int64_t oracle_expert_bytes_fmt(int fmt, int64_t D, int64_t F) {
  return 2 * fmt_bytes(fmt, F, D) + fmt_bytes(fmt, D, F);
}

int64_t oracle_expert_bytes(int64_t D, int64_t F) { return oracle_expert_bytes_fmt(0, D, F); }

/* SwiGLU expert applied to n input rows:
 *   h = SiLU(Wg x) * (Wu x),  y = Wd h   ([UDS] 5.3.7 steps 3-4). */
static void expert_ffn(int fmt, const uint8_t *blob, int64_t D, int64_t F, const double *const *xs,
                       double *const *ys, int64_t n) {
  const uint8_t *gq = blob, *uq = blob + fmt_bytes(fmt, F, D), *dq = uq + fmt_bytes(fmt, F, D);
  double *rowg = (double *)malloc(sizeof(double) * (size_t)D);
  double *rowu = (double *)malloc(sizeof(double) * (size_t)D);
  double *rowd = (double *)malloc(sizeof(double) * (size_t)F);
  double *h = (double *)malloc(sizeof(double) * (size_t)(F * n));
  int64_t bpr_d = fmt_bytes(fmt, 1, D), bpr_f = fmt_bytes(fmt, 1, F);
  for (int64_t f = 0; f < F; ++f) {
    fmt_dequantize(fmt, gq + f * bpr_d, 1, D, rowg);
    fmt_dequantize(fmt, uq + f * bpr_d, 1, D, rowu);
    for (int64_t i = 0; i < n; ++i) {
      double g = 0.0, u = 0.0;
      for (int64_t d = 0; d < D; ++d) { g += rowg[d] * xs[i][d]; u += rowu[d] * xs[i][d]; }
      h[i * F + f] = silu(g) * u;
    }
  }
  for (int64_t d = 0; d < D; ++d) {
    fmt_dequantize(fmt, dq + d * bpr_f, 1, F, rowd);
    for (int64_t i = 0; i < n; ++i) {
      double y = 0.0;
      for (int64_t f = 0; f < F; ++f) y += rowd[f] * h[i * F + f];
      ys[i][d] = y;
    }
  }
  free(rowg); free(rowu); free(rowd); free(h);
}

/* Dense SwiGLU with fp64 weights (the shared expert, [UDS] 5.3.4). */
static void dense_ffn(const double *wg, const double *wu, const double *wd, int64_t D, int64_t Fs,
                      const double *x, double *y) {
  double *h = (double *)malloc(sizeof(double) * (size_t)Fs);
  for (int64_t f = 0; f < Fs; ++f) {
    double g = 0.0, u = 0.0;
    for (int64_t d = 0; d < D; ++d) { g += wg[f * D + d] * x[d]; u += wu[f * D + d] * x[d]; }
    h[f] = silu(g) * u;
  }
  for (int64_t d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t f = 0; f < Fs; ++f) acc += wd[d * Fs + f] * h[f];
    y[d] = acc;
  }
  free(h);
}

/* ----------------------------------------------------------------- layer --- */

typedef struct {
  int fmt;
  int64_t T, D, E, F, Fs; int32_t k;
  const double *x; const uint8_t *const *experts;
  const double *sg, *su, *sd;
  const int32_t *offsets, *perm;
  const int64_t *used; int64_t n_used;
  double *y;   /* [T*k][D], indexed by pair t*k+j */
  double *ys;  /* [T][D] shared expert output */
  int tid, nthreads;
} layer_job;

/* Work items: the used experts (each applied to all its tokens), then the
 * shared expert once per token.  Thread tid takes items tid, tid+n, ... */
static void *layer_worker(void *p) {
  layer_job *j = (layer_job *)p;
  int64_t n_items = j->n_used + (j->Fs > 0 ? j->T : 0);
  for (int64_t it = j->tid; it < n_items; it += j->nthreads) {
    if (it < j->n_used) {
      int64_t e = j->used[it];
      int64_t n = j->offsets[e + 1] - j->offsets[e];
      const double **xs = (const double **)malloc(sizeof(double *) * (size_t)n);
      double **ys = (double **)malloc(sizeof(double *) * (size_t)n);
      for (int64_t r = 0; r < n; ++r) {
        int64_t pair = j->perm[j->offsets[e] + r];
        xs[r] = j->x + (pair / j->k) * j->D;
        ys[r] = j->y + pair * j->D;
      }
      expert_ffn(j->fmt, j->experts[e], j->D, j->F, xs, ys, n);
      free(xs); free(ys);
    } else {
      int64_t t = it - j->n_used;
      dense_ffn(j->sg, j->su, j->sd, j->D, j->Fs, j->x + t * j->D, j->ys + t * j->D);
    }
  }
  return NULL;
}

/* One routed MoE layer ([UDS] 5.3.2 and 5.3.7):
 *   out[t] = shared(x_t) + sum_{j<k} w[t][j] * expert_{ids[t][j]}(x_t),
 * summed in that order.  experts[e] points at expert e's packed gate|up|down
 * (may be NULL for an expert no token selects).  sg/su/sd: shared expert
 * weights (ignored when Fs == 0).  ids, w: from oracle_select.  y_pairs
 * [T*k][D] and y_shared [T][D] are optional outputs.  fmt: the routed
 * experts' format (0 = Q2_K, 1 = Q4_K).
 * Returns 0, or -1 when a selected expert's weights are missing. */
int oracle_moe_layer_fmt(int fmt, int64_t T, int64_t D, int64_t E, int64_t F, int64_t Fs, int32_t k,
                         const double *x, const uint8_t *const *experts, const double *sg,
                         const double *su, const double *sd, const int32_t *ids, const double *w,
                         double *out, double *y_pairs, double *y_shared, int nthreads) {
  if (T == 0) return 0;
  int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T * k));
  int64_t *used = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
  oracle_route(ids, T, k, E, counts, offsets, perm, NULL);
  int64_t n_used = 0;
  int bad = 0;
  for (int64_t e = 0; e < E; ++e)
    if (counts[e]) { used[n_used++] = e; if (!experts[e]) bad = 1; }
  double *y = y_pairs ? y_pairs : (double *)malloc(sizeof(double) * (size_t)(T * k * D));
  double *ys = y_shared ? y_shared : (double *)malloc(sizeof(double) * (size_t)(T * D));
  if (!bad) {
    if (Fs == 0) memset(ys, 0, sizeof(double) * (size_t)(T * D));
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    layer_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
      layer_job j = {fmt, T, D, E, F, Fs, k, x, experts, sg, su, sd, offsets, perm, used, n_used,
                     y, ys, t, nthreads};
      jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, layer_worker, &jobs[t]);
    layer_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    for (int64_t t = 0; t < T; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double acc = ys[t * D + d];
        for (int32_t j = 0; j < k; ++j) acc += w[t * k + j] * y[(t * k + j) * D + d];
        out[t * D + d] = acc;
      }
  }
  if (!y_pairs) free(y);
  if (!y_shared) free(ys);
  free(used); free(counts); free(offsets); free(perm);
  return bad ? -1 : 0;
}

/* The layer with Q2_K experts. */
int oracle_moe_layer(int64_t T, int64_t D, int64_t E, int64_t F, int64_t Fs, int32_t k,
                     const double *x, const uint8_t *const *experts, const double *sg,
                     const double *su, const double *sd, const int32_t *ids, const double *w,
                     double *out, double *y_pairs, double *y_shared, int nthreads) {
  return oracle_moe_layer_fmt(0, T, D, E, F, Fs, k, x, experts, sg, su, sd, ids, w, out, y_pairs,
                              y_shared, nthreads);
}

/* ------------------------------------------------------------ RMSNorm --- */

/* Round a double to the nearest bf16 value (ties to even), returned as the
 * bf16 bit pattern. */
uint16_t oracle_bf16_round(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000 : 0;
  int e = ilogb(v);
  if (e < -126) e = -126;          /* subnormal spacing */
  double ulp = ldexp(1.0, e - 7);  /* 8 significant bits */
  double r = nearbyint(v / ulp) * ulp; /* default rounding mode: ties to even */
  float f = (float)r;              /* exact: r has at most 9 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* r = x / sqrt(mean(x^2) + eps) with unit gain, rounded to bf16 (pages:
 * "Layer normalization (RMSNorm)" per layer; eps and gain as fixed by the
 * workload).  x fp32 [T][D] -> r_bf16 [T][D]. */
void oracle_rmsnorm_bf16(const float *x, int64_t T, int64_t D, double eps, uint16_t *r_bf16) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t d = 0; d < D; ++d) ss += (double)x[t * D + d] * (double)x[t * D + d];
    double inv = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t d = 0; d < D; ++d) r_bf16[t * D + d] = oracle_bf16_round((double)x[t * D + d] * inv);
  }
}
