// Row formats of the quantised experts for the integer decode kernels:
// fixed-point activation planes, each lane's part of a Q2_K or Q4_K row, and
// exact row . activation dot products with dp4a ("Understanding Dwarf Star",
// 3.3.3 Q2_K block, 2.3.2 Q4_K block, 2.8.1-2.8.2 dequantise on the fly).
//
// Included by the decode translation units; everything here is inline or a
// template in an unnamed namespace, so each unit has its own copy.
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace dsm {
namespace {

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------- fixed point planes --
// For a vector of nb blocks (nsb = 16 nb sub-blocks): nine planes of nsb words
// (hi0..3, lo0..3, SX) then nb steps.  Word i of hi (lo) for sub-block sb
// holds in byte c the high (low) byte of X_{16 sb + 4c + i}: the byte order of
// (codes >> 2i) & 0x03030303.  Within a plane the words are stored in the
// order lanes read them, so every vector load is conflict-free.
// Lane map of a row of nb blocks of SPB sub-blocks (nb = 32 SPL / SPB):
// LPB = SPB / SPL lanes per block; lane l takes block l / LPB, sub-blocks
// SPL (l % LPB) + i, i < SPL.
template <int SPL, int SPB = 16>
struct LaneMap {
  static constexpr int LPB = SPB / SPL;
  static constexpr int Q = SPL < 4 ? SPL : 4;
  __device__ static __forceinline__ int off(int lane, int i) {
    return (i / Q) * (32 * Q) + lane * Q + (i % Q);
  }
};

// One block per half-warp (lanes 0-15 and 16-31 convert one block each);
// lane & 15 holds sub-block s's 16 values.
template <int SPL>
__device__ __forceinline__ void digitize_block(const float v[16], int b, uint32_t *planes,
                                              float *steps, int nsb) {
  const int lane = threadIdx.x & 31, s = lane & 15;
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int e = 0;
  if (m > 0.f) frexpf(m, &e);  // m < 2^e
  const float inv = m > 0.f ? ldexpf(1.0f, 15 - e) : 0.f;
  uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
  int sx = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    int X = __float2int_rn(v[j] * inv);  // exact scaling by a power of two
    X = max(-32767, min(32767, X));
    sx += X;
    const int i = j & 3, c = 8 * (j >> 2);
    hi[i] |= ((uint32_t)(X >> 8) & 0xFFu) << c;
    lo[i] |= ((uint32_t)X & 0xFFu) << c;
  }
  const int lr = b * LaneMap<SPL>::LPB + s / SPL;  // the lane that reads this sub-block
  const int o = LaneMap<SPL>::off(lr, s % SPL);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    planes[i * nsb + o] = hi[i];
    planes[(4 + i) * nsb + o] = lo[i];
  }
  planes[8 * nsb + o] = (uint32_t)sx;
  if (s == 0) steps[b] = m > 0.f ? ldexpf(1.0f, e - 15) : 0.f;
}

template <int Q>
__device__ __forceinline__ void lds_words(const uint32_t *p, uint32_t w[Q]) {
  if (Q == 4) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if (Q == 2) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = p[0];
  }
}

// This lane's words of one Q2_K row (global): SPL code words, the scale bytes
// of its sub-blocks, and d/dmin.
template <int SPL>
struct RowPart {
  uint32_t codes[SPL];
  uint32_t scm[(SPL + 3) / 4];
  uint32_t dd;
};

template <int SPL>
__device__ __forceinline__ void load_row(const uint8_t *row, RowPart<SPL> &r) {
  const int lane = threadIdx.x & 31;
  constexpr int LPB = 16 / SPL;
  const uint8_t *blk = row + (lane / LPB) * QB;
  const int s0 = SPL * (lane % LPB);
  const uint32_t *cw = reinterpret_cast<const uint32_t *>(blk + 16 + 4 * s0);
#pragma unroll
  for (int i = 0; i < SPL; ++i) r.codes[i] = __ldcs(cw + i);  // streamed once
  if (SPL >= 4) {
    const uint32_t *sw = reinterpret_cast<const uint32_t *>(blk + s0);
#pragma unroll
    for (int i = 0; i < (SPL + 3) / 4; ++i) r.scm[i] = __ldcs(sw + i);
  } else {  // s0 is not 4-aligned: take the word holding the bytes
    const uint32_t w = __ldcs(reinterpret_cast<const uint32_t *>(blk + (s0 & ~3)));
    r.scm[0] = w >> (8 * (s0 & 3));
  }
  r.dd = __ldcs(reinterpret_cast<const uint32_t *>(blk + 80));
}

// sum over this lane's sub-blocks of (row) . (planes): exact integers, one
// conversion per lane.
template <int SPL>
__device__ __forceinline__ float row_dot(const RowPart<SPL> &r, const uint32_t *planes,
                                         const float *steps, int nsb) {
  using M = LaneMap<SPL>;
  constexpr int Q = M::Q;
  const int lane = threadIdx.x & 31;
  int accq = 0, accm = 0;
#pragma unroll
  for (int g = 0; g < SPL / Q; ++g) {
    uint32_t hi[4][Q], lo[4][Q], sx[Q];
    const int o = g * (32 * Q) + lane * Q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lds_words<Q>(planes + i * nsb + o, hi[i]);
      lds_words<Q>(planes + (4 + i) * nsb + o, lo[i]);
    }
    lds_words<Q>(planes + 8 * nsb + o, sx);
#pragma unroll
    for (int k = 0; k < Q; ++k) {
      const int sub = g * Q + k;
      const uint32_t codes = r.codes[sub];
      const int scm = (r.scm[sub >> 2] >> (8 * (sub & 3))) & 0xFF;
      const uint32_t q0 = codes & 0x03030303u, q1 = (codes >> 2) & 0x03030303u;
      const uint32_t q2 = (codes >> 4) & 0x03030303u, q3 = (codes >> 6) & 0x03030303u;
      int sh = __dp4a((int)q0, (int)hi[0][k], 0);
      sh = __dp4a((int)q1, (int)hi[1][k], sh);
      sh = __dp4a((int)q2, (int)hi[2][k], sh);
      sh = __dp4a((int)q3, (int)hi[3][k], sh);
      unsigned sl = __dp4a(q0, lo[0][k], 0u);
      sl = __dp4a(q1, lo[1][k], sl);
      sl = __dp4a(q2, lo[2][k], sl);
      sl = __dp4a(q3, lo[3][k], sl);
      accq += (scm & 15) * (sh * 256 + (int)sl);  // sc_s * sum_j q_j X_j
      accm += (scm >> 4) * (int)sx[k];            // m_s * sum_j X_j
    }
  }
  const float d = fp16_to_f32((uint16_t)(r.dd & 0xFFFF)), dmin = fp16_to_f32((uint16_t)(r.dd >> 16));
  return steps[lane / M::LPB] * fmaf(d, (float)accq, -dmin * (float)accm);
}

__device__ __forceinline__ void bf16x8(uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Butterfly sums of N independent values (all lanes end with the totals);
// the N shuffles of a level are independent, so they pipeline.
template <int N>
__device__ __forceinline__ void warp_sum_n(float v[N]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
}

// Warp totals of N values (N = 2, 4, 8) in 5 + N - 2 shuffles instead of
// 5 N: at each of the first levels a lane hands half of its running sums to
// its partner and keeps the other half.  Lane l ends with the total of
// v[l / (32 / N)].
template <int N>
__device__ __forceinline__ float warp_sum_spread(const float v[N]) {
  const int lane = threadIdx.x & 31;
  float cur[N];
#pragma unroll
  for (int i = 0; i < N; ++i) cur[i] = v[i];
  int n = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool hi = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = hi ? cur[i] : cur[n / 2 + i];
        const float keep = hi ? cur[n / 2 + i] : cur[i];
        cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
      n /= 2;
    } else {
      cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], o);
    }
  }
  return cur[0];
}

__device__ __forceinline__ int shfl(int v, int l) { return __shfl_sync(0xffffffffu, v, l); }
__device__ __forceinline__ float shflf(float v, int l) { return __shfl_sync(0xffffffffu, v, l); }

// This lane's words of one Q2_K row held in shared memory (layout as load_row).
template <int SPL>
__device__ __forceinline__ void load_row_s(const uint8_t *row, RowPart<SPL> &r) {
  const int lane = threadIdx.x & 31;
  constexpr int LPB = 16 / SPL;
  const uint8_t *blk = row + (lane / LPB) * QB;
  const int s0 = SPL * (lane % LPB);
  const uint32_t *cw = reinterpret_cast<const uint32_t *>(blk + 16 + 4 * s0);
#pragma unroll
  for (int i = 0; i < SPL; ++i) r.codes[i] = cw[i];
  if (SPL >= 4) {
    const uint32_t *sw = reinterpret_cast<const uint32_t *>(blk + s0);
#pragma unroll
    for (int i = 0; i < (SPL + 3) / 4; ++i) r.scm[i] = sw[i];
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(blk + (s0 & ~3));
    r.scm[0] = w >> (8 * (s0 & 3));
  }
  r.dd = *reinterpret_cast<const uint32_t *>(blk + 80);
}

// The lane's fixed-point activation words (the sub-blocks LaneMap gives it),
// held in registers for every row of a phase.
template <int SPL>
struct XReg {
  uint32_t hi[SPL][4], lo[SPL][4], sx[SPL];
  float step;
};

template <int SPL>
__device__ __forceinline__ void load_xreg(const uint32_t *planes, const float *steps, int nsb,
                                          XReg<SPL> &x) {
  using M = LaneMap<SPL>;
  constexpr int Q = M::Q;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int g = 0; g < SPL / Q; ++g) {
    const int o = g * (32 * Q) + lane * Q;
    uint32_t w[Q];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lds_words<Q>(planes + i * nsb + o, w);
#pragma unroll
      for (int k = 0; k < Q; ++k) x.hi[g * Q + k][i] = w[k];
      lds_words<Q>(planes + (4 + i) * nsb + o, w);
#pragma unroll
      for (int k = 0; k < Q; ++k) x.lo[g * Q + k][i] = w[k];
    }
    lds_words<Q>(planes + 8 * nsb + o, w);
#pragma unroll
    for (int k = 0; k < Q; ++k) x.sx[g * Q + k] = w[k];
  }
  x.step = steps[lane / M::LPB];
}

// row_dot with the activation words in registers.
template <int SPL>
__device__ __forceinline__ float row_dot_reg(const RowPart<SPL> &r, const XReg<SPL> &x) {
  int accq = 0, accm = 0;
#pragma unroll
  for (int sub = 0; sub < SPL; ++sub) {
    const uint32_t codes = r.codes[sub];
    const int scm = (r.scm[sub >> 2] >> (8 * (sub & 3))) & 0xFF;
    const uint32_t q0 = codes & 0x03030303u, q1 = (codes >> 2) & 0x03030303u;
    const uint32_t q2 = (codes >> 4) & 0x03030303u, q3 = (codes >> 6) & 0x03030303u;
    int sh = __dp4a((int)q0, (int)x.hi[sub][0], 0);
    sh = __dp4a((int)q1, (int)x.hi[sub][1], sh);
    sh = __dp4a((int)q2, (int)x.hi[sub][2], sh);
    sh = __dp4a((int)q3, (int)x.hi[sub][3], sh);
    unsigned sl = __dp4a(q0, x.lo[sub][0], 0u);
    sl = __dp4a(q1, x.lo[sub][1], sl);
    sl = __dp4a(q2, x.lo[sub][2], sl);
    sl = __dp4a(q3, x.lo[sub][3], sl);
    accq += (scm & 15) * (sh * 256 + (int)sl);  // sc_s * sum_j q_j X_j
    accm += (scm >> 4) * (int)x.sx[sub];        // m_s * sum_j X_j
  }
  const float d = fp16_to_f32((uint16_t)(r.dd & 0xFFFF)), dmin = fp16_to_f32((uint16_t)(r.dd >> 16));
  return x.step * fmaf(d, (float)accq, -dmin * (float)accm);
}

// A lane's part of one Q2_K row with the sub-block scales folded into the
// codes, for rows that meet several activation vectors: byte c of qs[s][i]
// is sc_s * q of weight 4 c + i of the lane's sub-block s (at most 45), byte
// s of mm the min m_s, and d, dmin as floats.  Its dot with an activation is
// the same integer sum as row_dot_reg's,
//   sum_s sc_s (256 sum_j q_j hi_j + sum_j q_j lo_j) = 256 sum qs.hi + sum qs.lo,
// so the result is bit-identical, with half the instructions per vector.
template <int SPL>
struct ScRow {
  uint32_t qs[SPL][4];
  uint32_t mm[(SPL + 3) / 4];
  float d, dmin;
};

template <int SPL>
__device__ __forceinline__ void load_scrow_s(const uint8_t *row, ScRow<SPL> &r) {
  RowPart<SPL> p;
  load_row_s<SPL>(row, p);
#pragma unroll
  for (int s = 0; s < SPL; ++s) {
    const uint32_t sc = (p.scm[s >> 2] >> (8 * (s & 3))) & 15u;
#pragma unroll
    for (int i = 0; i < 4; ++i) r.qs[s][i] = ((p.codes[s] >> (2 * i)) & 0x03030303u) * sc;
  }
#pragma unroll
  for (int w = 0; w < (SPL + 3) / 4; ++w) r.mm[w] = (p.scm[w] >> 4) & 0x0F0F0F0Fu;
  r.d = fp16_to_f32((uint16_t)(p.dd & 0xFFFF));
  r.dmin = fp16_to_f32((uint16_t)(p.dd >> 16));
}

template <int SPL>
__device__ __forceinline__ float scrow_dot(const ScRow<SPL> &r, const XReg<SPL> &x) {
  int ah = 0, accm = 0;
  unsigned al = 0u;
#pragma unroll
  for (int s = 0; s < SPL; ++s) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ah = __dp4a((int)r.qs[s][i], (int)x.hi[s][i], ah);
      al = __dp4a(r.qs[s][i], x.lo[s][i], al);
    }
    accm += (int)((r.mm[s >> 2] >> (8 * (s & 3))) & 0xFFu) * (int)x.sx[s];
  }
  const int accq = ah * 256 + (int)al;
  return x.step * fmaf(r.d, (float)accq, -r.dmin * (float)accm);
}

// ------------------------------------------------------------- Q4_K rows --
// "Understanding Dwarf Star", 2.3.2: a 144-byte block holds fp16 d and dmin,
// twelve bytes of 6-bit sub-block scales and mins, and 128 bytes of 4-bit
// codes; 8 sub-blocks of 32 weights.  Code word c of sub-block s (bytes
// 16 + 16 s + 4 c) holds weights 8 c + 2 b (low nibble of byte b) and
// 8 c + 2 b + 1 (high nibble), so (word >> 4 p) & 0x0F0F0F0F puts the codes
// of parity p in the four bytes.  The fixed point planes of a vector follow
// the Q2_K ones with seventeen planes per 32-weight sub-block: the high bytes
// of X for the weights of code word c and parity p in plane 2 c + p, the low
// bytes in plane 8 + 2 c + p, the sub-block sum of X in plane 16; then nb
// steps.  Sums are exact integers as for Q2_K; a sub-block's scaled sum
// (15 * 32767 * 32 * 63 at most) fits in 32 bits, a lane's total needs 64.

// One block per half-warp: lane & 15 holds weights 16 (lane & 15) .. + 15 of
// the block, i.e. half (lane & 1) of sub-block (lane & 15) / 2.
template <int SPL>
__device__ __forceinline__ void digitize_block4(const float v[16], int b, uint32_t *planes,
                                               float *steps, int nsb) {
  using M = LaneMap<SPL, 8>;
  const int lane = threadIdx.x & 31, s = (lane & 15) >> 1, half = lane & 1;
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int e = 0;
  if (m > 0.f) frexpf(m, &e);  // m < 2^e
  const float inv = m > 0.f ? ldexpf(1.0f, 15 - e) : 0.f;
  uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};  // [2 * (local word) + parity]
  int sx = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    int X = __float2int_rn(v[j] * inv);  // exact scaling by a power of two
    X = max(-32767, min(32767, X));
    sx += X;
    const int idx = 2 * (j >> 3) + (j & 1), c = 8 * ((j & 7) >> 1);
    hi[idx] |= ((uint32_t)(X >> 8) & 0xFFu) << c;
    lo[idx] |= ((uint32_t)X & 0xFFu) << c;
  }
  sx += __shfl_xor_sync(0xffffffffu, sx, 1);  // the other half of the sub-block
  const int lr = b * M::LPB + s / SPL;       // the lane that reads this sub-block
  const int o = M::off(lr, s % SPL);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    planes[(4 * half + i) * nsb + o] = hi[i];
    planes[(8 + 4 * half + i) * nsb + o] = lo[i];
  }
  if (half == 0) planes[16 * nsb + o] = (uint32_t)sx;
  if ((lane & 15) == 0) steps[b] = m > 0.f ? ldexpf(1.0f, e - 15) : 0.f;
}

// This lane's parts of one Q4_K row in shared memory: the code words of its
// SPL sub-blocks and the block header (d, dmin, the 6-bit fields).
template <int SPL>
struct RowPart4 {
  uint4 codes[SPL];
  uint4 hdr;
};

// The same from global memory (every byte read once: streaming loads).
template <int SPL>
__device__ __forceinline__ void load_row4(const uint8_t *row, RowPart4<SPL> &r) {
  const int lane = threadIdx.x & 31;
  constexpr int LPB = 8 / SPL;
  const uint8_t *blk = row + (lane / LPB) * Q4B;
  const int s0 = SPL * (lane % LPB);
#pragma unroll
  for (int i = 0; i < SPL; ++i) r.codes[i] = __ldcs(reinterpret_cast<const uint4 *>(blk + 16 + 16 * (s0 + i)));
  r.hdr = __ldcs(reinterpret_cast<const uint4 *>(blk));
}

template <int SPL>
__device__ __forceinline__ void load_row_s4(const uint8_t *row, RowPart4<SPL> &r) {
  const int lane = threadIdx.x & 31;
  constexpr int LPB = 8 / SPL;
  const uint8_t *blk = row + (lane / LPB) * Q4B;
  const int s0 = SPL * (lane % LPB);
#pragma unroll
  for (int i = 0; i < SPL; ++i) r.codes[i] = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * (s0 + i));
  r.hdr = *reinterpret_cast<const uint4 *>(blk);
}

template <int SPL>
struct XReg4 {
  uint32_t hi[SPL][8], lo[SPL][8], sx[SPL];
  float step;
};

template <int SPL>
__device__ __forceinline__ void load_xreg4(const uint32_t *planes, const float *steps, int nsb,
                                           XReg4<SPL> &x) {
  using M = LaneMap<SPL, 8>;
  constexpr int Q = M::Q;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int g = 0; g < SPL / Q; ++g) {
    const int o = g * (32 * Q) + lane * Q;
    uint32_t w[Q];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lds_words<Q>(planes + i * nsb + o, w);
#pragma unroll
      for (int k = 0; k < Q; ++k) x.hi[g * Q + k][i] = w[k];
      lds_words<Q>(planes + (8 + i) * nsb + o, w);
#pragma unroll
      for (int k = 0; k < Q; ++k) x.lo[g * Q + k][i] = w[k];
    }
    lds_words<Q>(planes + 16 * nsb + o, w);
#pragma unroll
    for (int k = 0; k < Q; ++k) x.sx[g * Q + k] = w[k];
  }
  x.step = steps[lane / M::LPB];
}

// sc_s * sum_j q_j X_j of one sub-block: 16 dp4a over the even and odd codes.
__device__ __forceinline__ int q4_sub_dot(const uint4 &codes, const uint32_t hi[8], const uint32_t lo[8]) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  int sh = 0;
  unsigned sl = 0u;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t q = (cw[c] >> (4 * p)) & 0x0F0F0F0Fu;
      sh = __dp4a((int)q, (int)hi[2 * c + p], sh);
      sl = __dp4a(q, lo[2 * c + p], sl);
    }
  return sh * 256 + (int)sl;  // sum_j q_j X_j
}

// Q4_K row . activation with the activation words in registers.
template <int SPL>
__device__ __forceinline__ float row_dot_reg4(const RowPart4<SPL> &r, const XReg4<SPL> &x) {
  const int lane = threadIdx.x & 31;
  const int s0 = SPL * (lane % (8 / SPL));
  long long accq = 0, accm = 0;
#pragma unroll
  for (int sub = 0; sub < SPL; ++sub) {
    const int sc = q4k_field(r.hdr, s0 + sub), mm = q4k_field(r.hdr, 8 + s0 + sub);
    accq += (long long)sc * q4_sub_dot(r.codes[sub], x.hi[sub], x.lo[sub]);
    accm += (long long)mm * (int)x.sx[sub];
  }
  const float d = fp16_to_f32((uint16_t)(r.hdr.x & 0xFFFF)), dmin = fp16_to_f32((uint16_t)(r.hdr.x >> 16));
  return x.step * fmaf(d, (float)accq, -dmin * (float)accm);
}

// The same with the activation planes read from shared memory.
template <int SPL>
__device__ __forceinline__ float row_dot4(const RowPart4<SPL> &r, const uint32_t *planes,
                                          const float *steps, int nsb) {
  XReg4<SPL> x;
  load_xreg4<SPL>(planes, steps, nsb, x);
  return row_dot_reg4<SPL>(r, x);
}

// Row formats of the one-token streaming kernel: bytes per block, weights
// per sub-block, fixed point planes per sub-block, and the lane's row parts,
// activation registers, loads and dots.
template <int SPL>
struct Q2Rows {
  static constexpr int BB = QB, SUB = 16, NPL = 9;
  using Row = RowPart<SPL>;
  using XR = XReg<SPL>;
  __device__ static __forceinline__ void digitize(const float v[16], int b, uint32_t *pl, float *st, int nsb) {
    digitize_block<SPL>(v, b, pl, st, nsb);
  }
  __device__ static __forceinline__ void load_x(const uint32_t *pl, const float *st, int nsb, XR &x) {
    load_xreg<SPL>(pl, st, nsb, x);
  }
  __device__ static __forceinline__ void load_s(const uint8_t *row, Row &r) { load_row_s<SPL>(row, r); }
  __device__ static __forceinline__ void load_g(const uint8_t *row, Row &r) { load_row<SPL>(row, r); }
  __device__ static __forceinline__ float dot_reg(const Row &r, const XR &x) { return row_dot_reg<SPL>(r, x); }
  __device__ static __forceinline__ float dot(const Row &r, const uint32_t *pl, const float *st, int nsb) {
    return row_dot<SPL>(r, pl, st, nsb);
  }
};

template <int SPL>
struct Q4Rows {
  static constexpr int BB = Q4B, SUB = 32, NPL = 17;
  using Row = RowPart4<SPL>;
  using XR = XReg4<SPL>;
  __device__ static __forceinline__ void digitize(const float v[16], int b, uint32_t *pl, float *st, int nsb) {
    digitize_block4<SPL>(v, b, pl, st, nsb);
  }
  __device__ static __forceinline__ void load_x(const uint32_t *pl, const float *st, int nsb, XR &x) {
    load_xreg4<SPL>(pl, st, nsb, x);
  }
  __device__ static __forceinline__ void load_s(const uint8_t *row, Row &r) { load_row_s4<SPL>(row, r); }
  __device__ static __forceinline__ void load_g(const uint8_t *row, Row &r) { load_row4<SPL>(row, r); }
  __device__ static __forceinline__ float dot_reg(const Row &r, const XR &x) { return row_dot_reg4<SPL>(r, x); }
  __device__ static __forceinline__ float dot(const Row &r, const uint32_t *pl, const float *st, int nsb) {
    return row_dot4<SPL>(r, pl, st, nsb);
  }
};

}  // namespace
}  // namespace dsm
