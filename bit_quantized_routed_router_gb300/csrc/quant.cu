// Q2_K and Q4_K quantiser and dequantiser kernels.
//
// Block format and the reading of "four evenly spaced levels between the
// block's min and max": "Understanding Dwarf Star", 3.3.3 "Q2_K: 2.625 Bits
// Per Element" and 2.3.5; layout restated in include/ds_moe.h.
#include "common.cuh"
#include "internal.h"

namespace dsm {
namespace {

__device__ __forceinline__ double h2d(int bits) {
  return (double)__half2float(__ushort_as_half((unsigned short)bits));
}

// One warp per super-block.  Lane l owns sub-block s = l % 16 and the half
// h = l / 16 of its 16 weights (8 weights).  Every scale decision is an exact
// comparison in fp64, so the encoding is a pure function of the input bits.
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ w, int64_t rows,
                                                       int64_t in_dim, int64_t nb,
                                                       uint8_t *__restrict__ out, unsigned *st) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (blk >= rows * nb) return;
  const int64_t r = blk / nb, b = blk % nb;
  const int s = lane & 15, h = lane >> 4;
  float v[8];
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int64_t c = b * QK + 16 * s + 8 * h + i;
    v[i] = c < in_dim ? w[r * in_dim + c] : 0.0f;  // zero padding
    ok = ok && (fabsf(v[i]) <= 65504.0f);           // also false for NaN
  }
  uint8_t *o = out + blk * QB;
  if (!__all_sync(0xffffffffu, ok)) {
    if (lane == 0) flag(st, ST_QUANT_INPUT);
    for (int i = lane; i < QB; i += 32) o[i] = 0;
    return;
  }
  float mn = 0.0f, mx = v[0];
#pragma unroll
  for (int i = 0; i < 8; ++i) { mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
  mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  const double neg_lo = -(double)mn, hi = (double)mx;

  // dmin: smallest fp16 with 15*dmin >= -lo_s for every sub-block.
  int lo_b = 0, hi_b = 0x7BFF;
  while (lo_b < hi_b) {
    int mid = (lo_b + hi_b) >> 1;
    if (__all_sync(0xffffffffu, 15.0 * h2d(mid) >= neg_lo)) hi_b = mid; else lo_b = mid + 1;
  }
  const int dmin_bits = lo_b;
  const double dmin = h2d(dmin_bits);
  int m = 0;
  while (m < 15 && (double)m * dmin < neg_lo) ++m;
  const double bs = (double)m * dmin;  // exact

  // d: smallest fp16 with 45*d - b_s >= hi_s for every sub-block (exact).
  lo_b = 0; hi_b = 0x7BFF;
  while (lo_b < hi_b) {
    int mid = (lo_b + hi_b) >> 1;
    if (__all_sync(0xffffffffu, 45.0 * h2d(mid) - bs >= hi)) hi_b = mid; else lo_b = mid + 1;
  }
  const int d_bits = lo_b;
  const double d = h2d(d_bits);
  int sc = 0;
  while (sc < 15 && 3.0 * d * (double)sc - bs < hi) ++sc;

  // codes: q = #{i in 1..3 : x >= (i - 1/2) d sc - b}, each threshold exact.
  uint32_t packed = 0;
  if (sc > 0) {
    const double t1 = 0.5 * d * (double)sc - bs, t2 = 1.5 * d * (double)sc - bs,
                 t3 = 2.5 * d * (double)sc - bs;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      double x = (double)v[i];
      uint32_t q = (x >= t1) + (x >= t2) + (x >= t3);
      packed |= q << (2 * i);
    }
  }
  // weights 16s + 8h + (0..7) -> bytes 16 + 4s + 2h (+1)
  o[16 + 4 * s + 2 * h] = (uint8_t)(packed & 0xFF);
  o[16 + 4 * s + 2 * h + 1] = (uint8_t)(packed >> 8);
  if (h == 0) o[s] = (uint8_t)(sc | (m << 4));
  if (lane == 0) {
    o[80] = (uint8_t)(d_bits & 0xFF);
    o[81] = (uint8_t)(d_bits >> 8);
    o[82] = (uint8_t)(dmin_bits & 0xFF);
    o[83] = (uint8_t)(dmin_bits >> 8);
  }
}

// One thread per weight: fp32(d*sc*q - dmin*m).  d*sc and dmin*m are exact in
// fp32 (an fp16 times a 4-bit integer), so the single fused multiply-add
// rounds the exact value once.
__global__ void dequantize_kernel(const uint8_t *__restrict__ q, int64_t rows, int64_t in_dim,
                                  int64_t nb, float *__restrict__ out) {
  const int64_t n = rows * in_dim;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / in_dim, c = i % in_dim;
    const uint8_t *blk = q + (r * nb + c / QK) * QB;
    const int j = (int)(c % QK), s = j >> 4;
    const float d = fp16_to_f32((uint16_t)(blk[80] | (blk[81] << 8)));
    const float dmin = fp16_to_f32((uint16_t)(blk[82] | (blk[83] << 8)));
    const int sc = blk[s] & 15, m = blk[s] >> 4;
    const int code = (blk[16 + (j >> 2)] >> (2 * (j & 3))) & 3;
    out[i] = __fmaf_rn(__fmul_rn(d, (float)sc), (float)code, -__fmul_rn(dmin, (float)m));
  }
}

// ---------------------------------------------------------------- Q4_K --
// "Understanding Dwarf Star", 2.3.2 "K-Quant Formats": 144-byte block, fp16
// d and dmin, 12 bytes of 6-bit sub-block scales and mins, 128 bytes of
// 4-bit codes, 8 sub-blocks of 32 weights (packing in include/ds_moe.h).

// One warp per super-block.  Lane l owns sub-block s = l / 4 and its
// quarter c = l % 4 (weights 32 s + 8 c + 0..7).  The same exact decisions
// as the Q2_K kernel with 15 levels and 6-bit scales and mins.
__global__ void __launch_bounds__(256) quantize_q4k_kernel(const float *__restrict__ w, int64_t rows,
                                                           int64_t in_dim, int64_t nb,
                                                           uint8_t *__restrict__ out, unsigned *st) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (blk >= rows * nb) return;
  const int64_t r = blk / nb, b = blk % nb;
  const int s = lane >> 2, c = lane & 3;
  float v[8];
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int64_t col = b * QK + 32 * s + 8 * c + i;
    v[i] = col < in_dim ? w[r * in_dim + col] : 0.0f;  // zero padding
    ok = ok && (fabsf(v[i]) <= 65504.0f);               // also false for NaN
  }
  uint8_t *o = out + blk * Q4B;
  if (!__all_sync(0xffffffffu, ok)) {
    if (lane == 0) flag(st, ST_QUANT_INPUT);
    for (int i = lane; i < Q4B; i += 32) o[i] = 0;
    return;
  }
  float mn = 0.0f, mx = v[0];
#pragma unroll
  for (int i = 0; i < 8; ++i) { mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
#pragma unroll
  for (int x = 1; x < 4; x <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, x));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
  }
  const double neg_lo = -(double)mn, hi = (double)mx;

  // dmin: smallest fp16 with 63*dmin >= -lo_s for every sub-block.
  int lo_b = 0, hi_b = 0x7BFF;
  while (lo_b < hi_b) {
    int mid = (lo_b + hi_b) >> 1;
    if (__all_sync(0xffffffffu, 63.0 * h2d(mid) >= neg_lo)) hi_b = mid; else lo_b = mid + 1;
  }
  const int dmin_bits = lo_b;
  const double dmin = h2d(dmin_bits);
  int m = 0;
  while (m < 63 && (double)m * dmin < neg_lo) ++m;
  const double bs = (double)m * dmin;  // exact

  // d: smallest fp16 with 945*d - b_s >= hi_s for every sub-block (exact).
  lo_b = 0; hi_b = 0x7BFF;
  while (lo_b < hi_b) {
    int mid = (lo_b + hi_b) >> 1;
    if (__all_sync(0xffffffffu, 945.0 * h2d(mid) - bs >= hi)) hi_b = mid; else lo_b = mid + 1;
  }
  const int d_bits = lo_b;
  const double d = h2d(d_bits);
  int sc = 0;
  while (sc < 63 && 15.0 * d * (double)sc - bs < hi) ++sc;

  // codes: q = #{i in 1..15 : x >= (i - 1/2) d sc - b}, each threshold exact.
  uint32_t packed = 0;
  if (sc > 0) {
    const double step = d * (double)sc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const double x = (double)v[i];
      uint32_t q = 0;
      for (int t = 1; t <= 15; ++t) q += x >= ((double)t - 0.5) * step - bs;
      packed |= q << (4 * i);
    }
  }
  // weights 32 s + 8 c + (0..7) -> bytes 16 + 16 s + 4 c (+0..3)
  *reinterpret_cast<uint32_t *>(o + 16 + 16 * s + 4 * c) = packed;
  // 6-bit fields: sc_s is field s, m_s field 8 + s, field i at bits [6i, 6i+6)
  uint64_t f_lo = 0;
  uint32_t f_hi = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint64_t sct = (uint64_t)__shfl_sync(0xffffffffu, sc, 4 * t);
    const uint64_t mt = (uint64_t)__shfl_sync(0xffffffffu, m, 4 * t);
    f_lo |= sct << (6 * t);             // bits 0..47
    const int p = 48 + 6 * t;           // bits 48..95
    if (p + 6 <= 64) f_lo |= mt << p;
    else if (p >= 64) f_hi |= (uint32_t)(mt << (p - 64));
    else { f_lo |= mt << p; f_hi |= (uint32_t)(mt >> (64 - p)); }
  }
  if (lane == 0) {
    uint32_t *o32 = reinterpret_cast<uint32_t *>(o);
    o32[0] = (uint32_t)d_bits | ((uint32_t)dmin_bits << 16);
    o32[1] = (uint32_t)f_lo;
    o32[2] = (uint32_t)(f_lo >> 32);
    o32[3] = f_hi;
  }
}

// Sub-block scale (s < 8) or min (s >= 8) of a Q4_K block.
__device__ __forceinline__ int q4k_field_bytes(const uint8_t *blk, int i) {
  const int p = 6 * i;
  const uint32_t lo = blk[4 + (p >> 3)], hi = (p >> 3) + 5 < 16 ? blk[5 + (p >> 3)] : 0u;
  return (int)(((lo | (hi << 8)) >> (p & 7)) & 63u);
}

// One thread per weight, fp32(d*sc*q - dmin*m) rounded once (as for Q2_K:
// d*sc and dmin*m are exact in fp32, an fp16 times a 6-bit integer).
__global__ void dequantize_q4k_kernel(const uint8_t *__restrict__ q, int64_t rows, int64_t in_dim,
                                      int64_t nb, float *__restrict__ out) {
  const int64_t n = rows * in_dim;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / in_dim, c = i % in_dim;
    const uint8_t *blk = q + (r * nb + c / QK) * Q4B;
    const int j = (int)(c % QK), s = j >> 5;
    const float d = fp16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    const float dmin = fp16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const int sc = q4k_field_bytes(blk, s), m = q4k_field_bytes(blk, 8 + s);
    const int code = (blk[16 + (j >> 1)] >> (4 * (j & 1))) & 15;
    out[i] = __fmaf_rn(__fmul_rn(d, (float)sc), (float)code, -__fmul_rn(dmin, (float)m));
  }
}

}  // namespace

cudaError_t launch_quantize(int fmt, const float *w, int64_t rows, int64_t in_dim, uint8_t *out,
                            cudaStream_t s) {
  const int64_t nb = (in_dim + QK - 1) / QK;
  const int64_t blocks = rows * nb;
  if (blocks == 0) return cudaSuccess;
  const int64_t grid = (blocks + 7) / 8;
  if (fmt == DS_Q4_K)
    quantize_q4k_kernel<<<(unsigned)grid, 256, 0, s>>>(w, rows, in_dim, nb, out, status_word());
  else
    quantize_kernel<<<(unsigned)grid, 256, 0, s>>>(w, rows, in_dim, nb, out, status_word());
  return cudaGetLastError();
}

cudaError_t launch_dequantize(int fmt, const uint8_t *q, int64_t rows, int64_t in_dim, float *out,
                              cudaStream_t s) {
  const int64_t nb = (in_dim + QK - 1) / QK;
  const int64_t n = rows * in_dim;
  if (n == 0) return cudaSuccess;
  int64_t grid = (n + 255) / 256;
  if (grid > NUM_SMS * 32) grid = NUM_SMS * 32;
  if (fmt == DS_Q4_K) dequantize_q4k_kernel<<<(unsigned)grid, 256, 0, s>>>(q, rows, in_dim, nb, out);
  else dequantize_kernel<<<(unsigned)grid, 256, 0, s>>>(q, rows, in_dim, nb, out);
  return cudaGetLastError();
}

}  // namespace dsm
