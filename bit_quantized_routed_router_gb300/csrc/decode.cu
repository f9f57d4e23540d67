// Grouped dequantising GEMVs (gate/up with SwiGLU, then down), the weighted
// combine and the RMSNorm step of the stack.
//
// "Understanding Dwarf Star", 2.8.2 "Grouped Matrix Multiplication": load a
// 256-weight block, its scale, min and sub-block scales, dequantise, multiply
// by the 256 activations and accumulate; 5.3.7 "The MoE Kernel in Metal":
// gate projection -> activation -> down projection, multiply by the router
// weight and accumulate; 5.3.4: the shared expert runs for every token.
#include "common.cuh"
#include "internal.h"

namespace dsm {
namespace {

constexpr int NT = 4;     // tokens per staged group
constexpr int RPB = 32;   // output rows per block (8 warps x 4)

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

struct GemvArgs {
  const uint8_t *experts;
  int64_t expert_bytes, off_a, off_b;  // gate|up (GU) or down (DN) offsets in a blob
  const int32_t *slot;                 // residency: [E] cache slot or -1 (host copy); null: experts
  const uint8_t *cache, *host;
  const uint16_t *sh_a, *sh_b;         // shared expert rows (bf16): gate, up | down
  const void *in;                      // GU: x [T][D] (x_dtype); DN: h [T*k][F] fp32
  const float *in_shared;              // DN: hs [T][Fs]
  float *out;                          // GU: h [T*k][F]; DN: y [T*k][D]
  float *out_shared;                   // GU: hs [T][Fs]; DN: ys [T][D]
  const int32_t *offsets, *perm, *used;
  int64_t T;
  int k, E, D, F, Fs;
  int n_slots;
};

// float4 slot swizzle: chunk c of a staged row lives at c ^ ((c >> 3) & 7),
// so the 8 lanes of a quarter-warp reading chunks 4*sb + jj (Q2_K rows) or
// 2*lane (+1) (bf16 rows) hit 8 different 16-byte bank groups.
__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 3) & 7); }

template <typename TX>
__device__ __forceinline__ float4 load_in4(const TX *p);
template <>
__device__ __forceinline__ float4 load_in4<float>(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 load_in4<uint16_t>(const uint16_t *p) {
  uint2 v = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
}

// Partial dot products of one Q2_K row with nt staged inputs (this lane's
// sub-blocks sb = lane + 32 i).  w_j = d*sc*q_j - dmin*m is formed exactly in
// fp32 by one fused multiply-add, then multiplied into each input.
template <int NTOK>
__device__ __forceinline__ void q2k_row_dot(const uint8_t *__restrict__ row, int in_dim,
                                            const float4 *__restrict__ xs, int stride4, int nt,
                                            float acc[NTOK]) {
  const int lane = threadIdx.x & 31;
  const int nsb = in_dim >> 4;
  for (int sb = lane; sb < nsb; sb += 32) {
    const uint8_t *blk = row + (sb >> 4) * QB;
    const int s = sb & 15;
    const uint32_t codes = *reinterpret_cast<const uint32_t *>(blk + 16 + 4 * s);
    const uint32_t dd = *reinterpret_cast<const uint32_t *>(blk + 80);
    const int scm = blk[s];
    const float dsc = fp16_to_f32((uint16_t)(dd & 0xFFFF)) * (float)(scm & 15);
    const float dmm = fp16_to_f32((uint16_t)(dd >> 16)) * (float)(scm >> 4);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = __fmaf_rn(dsc, (float)((codes >> (2 * (4 * jj + i))) & 3u), -dmm);
      const int slot = swz(4 * sb + jj);
#pragma unroll
      for (int t = 0; t < NTOK; ++t) {
        if (t < nt) {
          const float4 xv = xs[t * stride4 + slot];
          acc[t] = fmaf(w[0], xv.x, acc[t]);
          acc[t] = fmaf(w[1], xv.y, acc[t]);
          acc[t] = fmaf(w[2], xv.z, acc[t]);
          acc[t] = fmaf(w[3], xv.w, acc[t]);
        }
      }
    }
  }
}

// Partial dot products of NR Q4_K rows ("Understanding Dwarf Star", 2.3.2:
// 8 sub-blocks of 32 weights, 6-bit scales and mins, 4-bit codes) with nt
// staged inputs; this lane's sub-blocks sb = lane + 32 i.  The code and
// header loads of all NR rows for one sub-block are issued
// before their use.  Weights formed exactly as for Q2_K.
template <int NR, int NTOK>
__device__ __forceinline__ void q4k_rows_dot(const uint8_t *const *rows, int in_dim,
                                             const float4 *__restrict__ xs, int stride4, int nt,
                                             float (*acc)[NTOK]) {
  const int lane = threadIdx.x & 31;
  const int nsb = in_dim >> 5;
  for (int sb = lane; sb < nsb; sb += 32) {
    const int s = sb & 7;
    uint4 codes[NR], hdr[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint8_t *blk = rows[r] + (sb >> 3) * Q4B;
      codes[r] = __ldg(reinterpret_cast<const uint4 *>(blk + 16 + 16 * s));
      hdr[r] = __ldg(reinterpret_cast<const uint4 *>(blk));  // d, dmin, 12 field bytes
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int sc = q4k_field(hdr[r], s), mm = q4k_field(hdr[r], 8 + s);
      const float dsc = fp16_to_f32((uint16_t)(hdr[r].x & 0xFFFF)) * (float)sc;
      const float dmm = fp16_to_f32((uint16_t)(hdr[r].x >> 16)) * (float)mm;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t cw = jj < 2 ? codes[r].x : jj < 4 ? codes[r].y : jj < 6 ? codes[r].z : codes[r].w;
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = __fmaf_rn(dsc, (float)((cw >> (4 * (4 * (jj & 1) + i))) & 15u), -dmm);
        const int slot = swz(8 * sb + jj);
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          if (t < nt) {
            const float4 xv = xs[t * stride4 + slot];
            acc[r][t] = fmaf(w[0], xv.x, acc[r][t]);
            acc[r][t] = fmaf(w[1], xv.y, acc[r][t]);
            acc[r][t] = fmaf(w[2], xv.z, acc[r][t]);
            acc[r][t] = fmaf(w[3], xv.w, acc[r][t]);
          }
        }
      }
    }
  }
}

// Two rows (gate and up) in the format FMT.
template <int FMT, int NTOK>
__device__ __forceinline__ void q_rows_dot2(const uint8_t *__restrict__ ra, const uint8_t *__restrict__ rb,
                                            int in_dim, const float4 *__restrict__ xs, int stride4,
                                            int nt, float acc_a[NTOK], float acc_b[NTOK]) {
  if (FMT == DS_Q4_K) {
    float acc[2][NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) { acc[0][t] = acc_a[t]; acc[1][t] = acc_b[t]; }
    const uint8_t *rows[2] = {ra, rb};
    q4k_rows_dot<2, NTOK>(rows, in_dim, xs, stride4, nt, acc);
#pragma unroll
    for (int t = 0; t < NTOK; ++t) { acc_a[t] = acc[0][t]; acc_b[t] = acc[1][t]; }
  } else {
    q2k_row_dot<NTOK>(ra, in_dim, xs, stride4, nt, acc_a);
    q2k_row_dot<NTOK>(rb, in_dim, xs, stride4, nt, acc_b);
  }
}

// One row in the format FMT.
template <int FMT, int NTOK>
__device__ __forceinline__ void q_row_dot1(const uint8_t *__restrict__ ra, int in_dim,
                                           const float4 *__restrict__ xs, int stride4, int nt,
                                           float acc_a[NTOK]) {
  if (FMT == DS_Q4_K) {
    float acc[1][NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) acc[0][t] = acc_a[t];
    const uint8_t *rows[1] = {ra};
    q4k_rows_dot<1, NTOK>(rows, in_dim, xs, stride4, nt, acc);
#pragma unroll
    for (int t = 0; t < NTOK; ++t) acc_a[t] = acc[0][t];
  } else {
    q2k_row_dot<NTOK>(ra, in_dim, xs, stride4, nt, acc_a);
  }
}

// Same for a bf16 row (the shared expert); lane covers elements 8*lane + 256 i.
template <int NTOK>
__device__ __forceinline__ void bf16_row_dot(const uint16_t *__restrict__ row, int in_dim,
                                             const float4 *__restrict__ xs, int stride4, int nt,
                                             float acc[NTOK]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 4
  for (int d = 8 * lane; d < in_dim; d += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + d));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    float w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = __uint_as_float(wv[i] << 16);
      w[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
    }
    const int c0 = swz(d >> 2), c1 = swz((d >> 2) + 1);
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      if (t < nt) {
        const float4 a = xs[t * stride4 + c0], b = xs[t * stride4 + c1];
        acc[t] = fmaf(w[0], a.x, acc[t]); acc[t] = fmaf(w[1], a.y, acc[t]);
        acc[t] = fmaf(w[2], a.z, acc[t]); acc[t] = fmaf(w[3], a.w, acc[t]);
        acc[t] = fmaf(w[4], b.x, acc[t]); acc[t] = fmaf(w[5], b.y, acc[t]);
        acc[t] = fmaf(w[6], b.z, acc[t]); acc[t] = fmaf(w[7], b.w, acc[t]);
      }
    }
  }
}

// grid.x: blocks of RPB output rows; grid.y: expert slot (used[slot]), the
// last y being the shared expert when Fs > 0.  Each block walks its slot's
// tokens in groups of NT, staging their inputs in shared memory as fp32.
template <int MODE, typename TX, int FMT>
__global__ void __launch_bounds__(256) grouped_gemv_kernel(GemvArgs a) {
  extern __shared__ float4 xs[];
  const int slot = blockIdx.y;
  const bool shared = slot == a.n_slots;
  int e = 0, n_tok = 0, base = 0;
  if (!shared) {
    if (slot >= a.used[a.E]) return;
    e = a.used[slot];
    base = a.offsets[e];
    n_tok = a.offsets[e + 1] - base;
  } else {
    n_tok = (int)a.T;
  }
  const int in_dim = MODE == MODE_GATEUP ? a.D : (shared ? a.Fs : a.F);
  const int out_rows = MODE == MODE_GATEUP ? (shared ? a.Fs : a.F) : a.D;
  const int r0 = blockIdx.x * RPB;
  if (r0 >= out_rows) return;
  const int stride4 = in_dim >> 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the expert's bytes: its cache slot, the host copy (ordinary loads) or
  // the experts array; the same bytes either way
  const int es = a.slot ? __ldg(a.slot + e) : 0;
  const uint8_t *blob = !a.slot ? a.experts + (int64_t)e * a.expert_bytes
                        : es >= 0 ? a.cache + (int64_t)es * a.expert_bytes
                                  : a.host + (int64_t)e * a.expert_bytes;
  const int64_t row_bytes = (int64_t)((in_dim + QK - 1) / QK) * (FMT == DS_Q4_K ? Q4B : QB);

  for (int g0 = 0; g0 < n_tok; g0 += NT) {
    const int nt = min(NT, n_tok - g0);
    __syncthreads();
    for (int i = threadIdx.x; i < nt * stride4; i += blockDim.x) {
      const int t = i / stride4, c = i % stride4;
      float4 v;
      if (MODE == MODE_GATEUP) {
        const int64_t tok = shared ? (int64_t)(g0 + t) : (int64_t)(a.perm[base + g0 + t] / a.k);
        v = load_in4<TX>((const TX *)a.in + tok * a.D + 4 * c);
      } else {
        const float *src = shared ? a.in_shared + (int64_t)(g0 + t) * a.Fs
                                  : (const float *)a.in + (int64_t)(base + g0 + t) * a.F;
        v = *reinterpret_cast<const float4 *>(src + 4 * c);
      }
      xs[t * stride4 + swz(c)] = v;
    }
    __syncthreads();
    for (int r = r0 + warp; r < min(r0 + RPB, out_rows); r += 8) {
      if (MODE == MODE_GATEUP) {
        float g[NT] = {}, u[NT] = {};
        if (shared) {
          bf16_row_dot<NT>(a.sh_a + (int64_t)r * a.D, in_dim, xs, stride4, nt, g);
          bf16_row_dot<NT>(a.sh_b + (int64_t)r * a.D, in_dim, xs, stride4, nt, u);
        } else {
          q_rows_dot2<FMT, NT>(blob + a.off_a + r * row_bytes, blob + a.off_b + r * row_bytes, in_dim,
                               xs, stride4, nt, g, u);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float gs = warp_sum(g[t]), us = warp_sum(u[t]);
          if (lane == 0 && t < nt) {
            const float h = silu(gs) * us;
            if (shared) a.out_shared[(int64_t)(g0 + t) * a.Fs + r] = h;
            else a.out[(int64_t)(base + g0 + t) * a.F + r] = h;
          }
        }
      } else {
        float y[NT] = {};
        if (shared) bf16_row_dot<NT>(a.sh_a + (int64_t)r * a.Fs, in_dim, xs, stride4, nt, y);
        else q_row_dot1<FMT, NT>(blob + a.off_a + r * row_bytes, in_dim, xs, stride4, nt, y);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float ys = warp_sum(y[t]);
          if (lane == 0 && t < nt) {
            if (shared) a.out_shared[(int64_t)(g0 + t) * a.D + r] = ys;
            else a.out[(int64_t)(base + g0 + t) * a.D + r] = ys;
          }
        }
      }
    }
  }
}

// out[t][d] (+)= ys[t][d] + sum_j w[t][j] * y[pos[t*k+j]][d], in slot order.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ ys,
                                                      const float *__restrict__ y,
                                                      const float *__restrict__ w,
                                                      const int32_t *__restrict__ pos, int64_t T,
                                                      int D, int k, int has_shared,
                                                      int accumulate, float *__restrict__ out) {
  const int d4 = D >> 2;
  const int64_t n = T * d4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / d4;
    const int c = (int)(i % d4);
    float4 acc = has_shared ? reinterpret_cast<const float4 *>(ys + t * D)[c]
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float wj = w[t * k + j];
      const float4 v = reinterpret_cast<const float4 *>(y + (int64_t)pos[t * k + j] * D)[c];
      acc.x = fmaf(wj, v.x, acc.x); acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z); acc.w = fmaf(wj, v.w, acc.w);
    }
    float4 *o = reinterpret_cast<float4 *>(out + t * D) + c;
    if (accumulate) {
      float4 r = *o;
      acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
    }
    *o = acc;
  }
}

// bf16(x / sqrt(mean(x^2) + eps)); one block per token.
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float *__restrict__ x, int D,
                                                           float eps, uint16_t *__restrict__ out) {
  __shared__ float red[8];
  const float *xr = x + (int64_t)blockIdx.x * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) ss = fmaf(xr[d], xr[d], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float inv = 1.0f / sqrtf(tot / (float)D + eps);
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    out[(int64_t)blockIdx.x * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(xr[d] * inv));
}

template <int MODE, typename TX, int FMT>
cudaError_t launch_gemv1(const GemvArgs &a, int out_rows_max, int in_dim_max, cudaStream_t s) {
  // a block stages at most min(T, NT) tokens (no slot has more than T)
  const size_t smem = (size_t)std::min<int64_t>(a.T, NT) * in_dim_max * sizeof(float);
  static OncePerDevice once;
  auto kern = grouped_gemv_kernel<MODE, TX, FMT>;
  cudaError_t e = once_per_device(once, [&]() {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (e != cudaSuccess) return e;
  dim3 g((out_rows_max + RPB - 1) / RPB, a.n_slots + (a.Fs > 0 ? 1 : 0));
  kern<<<g, 256, smem, s>>>(a);
  return cudaGetLastError();
}

template <int MODE, typename TX>
cudaError_t launch_gemv(int fmt, const GemvArgs &a, int out_rows_max, int in_dim_max, cudaStream_t s) {
  return fmt == DS_Q4_K ? launch_gemv1<MODE, TX, DS_Q4_K>(a, out_rows_max, in_dim_max, s)
                        : launch_gemv1<MODE, TX, DS_Q2_K>(a, out_rows_max, in_dim_max, s);
}

}  // namespace

cudaError_t launch_decode_ffn(const Shape &sh, const ds_moe_weights &W, const void *x,
                              const Work &wk, cudaStream_t s, const Residency *res) {
  GemvArgs a{};
  a.experts = W.experts;
  a.expert_bytes = sh.expert_bytes();
  if (res) {
    a.slot = res->slot;
    a.cache = res->cache;
    a.host = res->host;
  }
  a.offsets = wk.offsets;
  a.perm = wk.perm;
  a.used = wk.used;
  a.T = wk.T;
  a.k = sh.k; a.E = sh.E; a.D = sh.D; a.F = sh.F; a.Fs = sh.Fs;
  a.n_slots = (int)std::min<int64_t>((int64_t)sh.E, wk.T * sh.k);
  // gate/up + SwiGLU
  a.off_a = 0;
  a.off_b = sh.gate_bytes();
  a.sh_a = W.shared_gate;
  a.sh_b = W.shared_up;
  a.in = x;
  a.out = wk.h;
  a.out_shared = wk.hs;
  cudaError_t err;
  const int rows1 = std::max(sh.F, sh.Fs);
  if (sh.x_dtype == DS_BF16) err = launch_gemv<MODE_GATEUP, uint16_t>(sh.fmt, a, rows1, sh.D, s);
  else err = launch_gemv<MODE_GATEUP, float>(sh.fmt, a, rows1, sh.D, s);
  if (err != cudaSuccess) return err;
  // down
  a.off_a = 2 * sh.gate_bytes();
  a.off_b = 0;
  a.sh_a = W.shared_down;
  a.sh_b = nullptr;
  a.in = wk.h;
  a.in_shared = wk.hs;
  a.out = wk.y;
  a.out_shared = wk.ys;
  return launch_gemv<MODE_DOWN, float>(sh.fmt, a, sh.D, std::max(sh.F, sh.Fs), s);
}

cudaError_t launch_combine(const Shape &sh, const Work &wk, float *out, bool accumulate,
                           cudaStream_t s) {
  const int64_t n = wk.T * (sh.D / 4);
  int64_t grid = (n + 255) / 256;
  if (grid > NUM_SMS * 16) grid = NUM_SMS * 16;
  combine_kernel<<<(unsigned)grid, 256, 0, s>>>(wk.ys, wk.y, wk.w, wk.pos, wk.T, sh.D, sh.k,
                                                sh.Fs > 0, accumulate ? 1 : 0, out);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const float *x, int64_t T, int D, float eps, uint16_t *out,
                                cudaStream_t s) {
  rmsnorm_bf16_kernel<<<(unsigned)T, 256, 0, s>>>(x, D, eps, out);
  return cudaGetLastError();
}

}  // namespace dsm
