/* Seeded synthetic-input generator: the counter-based core shared by the
 * host (gen/dsgen_host.c) and device (gen/dsgen_cuda.cu) fills.
 *
 * This module produces the synthetic activations and weights that both the
 * oracle and the CUDA path consume.  It contains no part of the MoE method's
 * arithmetic (no quantisation, routing, FFN or combine): only random numbers
 * and the fp32 -> bf16 storage conversion of generated values.
 *
 * Generator definition
 *   Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *   easy as 1, 2, 3", SC'11), key (k0, k1), counter (c0, c1, c2, c3).
 *   Each generated element uses one Philox call:
 *     key     = (seed, layer)
 *     counter = (idx & 0xffffffff, idx >> 32, sub, tensor)
 *   where idx is the element's row-major index inside its tensor, sub is the
 *   expert index (weights) or the resample attempt (activations), and tensor
 *   is one of the DSGEN_T_* ids below.
 *
 *   normal(sigma): S = sum of the eight 16-bit halves of the four outputs
 *     (Irwin-Hall of order 8 on 16-bit uniforms, integer-exact), value =
 *     fp32( (float)(S - 262140) * c ), with c = fp32(sigma*sqrt(12/8)/65536)
 *     computed once on the host.  Mean 0, standard deviation sigma
 *     (to 2^-32 relative), support bounded by +-4.9 sigma.
 *   uniform(a): u = r0 >> 8 (24 bits), value = fp32( (float)(2u - (2^24-1)) * c )
 *     with c = fp32(a / 2^24): symmetric on (-a, a).
 *   Every step is an exact integer operation or a single IEEE fp32
 *   multiply, so host and device produce identical bits.
 */
#ifndef DSGEN_CORE_H
#define DSGEN_CORE_H
#include <stdint.h>

#if defined(__CUDACC__)
#define DSGEN_HD __host__ __device__ __forceinline__
#else
#define DSGEN_HD static inline
#endif

enum {
  DSGEN_T_X = 1,            /* activations x[T][D]                       */
  DSGEN_T_ROUTER_W = 2,     /* router weights [E][D]                     */
  DSGEN_T_ZIPF_PERM = 3,    /* Fisher-Yates draws for the popularity bias */
  DSGEN_T_SHARED_GATE = 4,  /* shared expert gate [Fs][D]                */
  DSGEN_T_SHARED_UP = 5,    /* shared expert up   [Fs][D]                */
  DSGEN_T_SHARED_DOWN = 6,  /* shared expert down [D][Fs]                */
  DSGEN_T_EXPERT_GATE = 7,  /* routed expert gate [F][D], sub = expert   */
  DSGEN_T_EXPERT_UP = 8,    /* routed expert up   [F][D], sub = expert   */
  DSGEN_T_EXPERT_DOWN = 9   /* routed expert down [D][F], sub = expert   */
};

DSGEN_HD void dsgen_mulhilo(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

/* Philox4x32 with 10 rounds; multipliers and Weyl key increments as
 * published by Salmon et al. (SC'11). */
DSGEN_HD void dsgen_philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                  uint32_t k0, uint32_t k1, uint32_t out[4]) {
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    dsgen_mulhilo(0xD2511F53u, c0, &hi0, &lo0);
    dsgen_mulhilo(0xCD9E8D57u, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

DSGEN_HD void dsgen_draw(uint32_t seed, uint32_t layer, uint32_t tensor, uint32_t sub,
                         uint64_t idx, uint32_t out[4]) {
  dsgen_philox4x32_10((uint32_t)idx, (uint32_t)(idx >> 32), sub, tensor, seed, layer, out);
}

DSGEN_HD float dsgen_normal(uint32_t seed, uint32_t layer, uint32_t tensor, uint32_t sub,
                            uint64_t idx, float c) {
  uint32_t r[4];
  dsgen_draw(seed, layer, tensor, sub, idx, r);
  int32_t s = 0;
  for (int i = 0; i < 4; ++i) s += (int32_t)(r[i] & 0xFFFFu) + (int32_t)(r[i] >> 16);
  float v = (float)(s - 262140); /* exact: |s - 262140| < 2^19 */
  return v * c;
}

DSGEN_HD float dsgen_uniform(uint32_t seed, uint32_t layer, uint32_t tensor, uint32_t sub,
                             uint64_t idx, float c) {
  uint32_t r[4];
  dsgen_draw(seed, layer, tensor, sub, idx, r);
  int32_t u = (int32_t)(r[0] >> 8);
  float v = (float)(2 * u - 16777215); /* exact: odd, |v| < 2^24 */
  return v * c;
}

/* fp32 -> bf16 storage, round to nearest even (inputs here are finite). */
DSGEN_HD uint16_t dsgen_f32_to_bf16(float f) {
  union { float f; uint32_t u; } cv;
  cv.f = f;
  uint32_t u = cv.u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#endif
