// Router logits, top-k selection and the expert route.
//
// "Understanding Dwarf Star", 5.3.2 "The MoE Architecture": router(x) =
// softmax(x W_router); the top-k experts by router probability are used and
// weighted by it; 5.3.7: "complex indexing required for sparse expert
// selection" -- here a histogram, an exclusive scan and a stable permutation
// that groups each expert's tokens contiguously.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsm {
namespace {

constexpr int ROUTE_CHUNK = 1024;  // pairs per permutation chunk

template <typename T>
__device__ __forceinline__ void load8(const T *p, float v[8]);

template <>
__device__ __forceinline__ void load8<float>(const float *p, float v[8]) {
  float4 a = *reinterpret_cast<const float4 *>(p);
  float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t *p, float v[8]) {
  uint4 a = *reinterpret_cast<const uint4 *>(p);
  uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// logits[t][e] = sum_d x[t][d] * Wr[e][d] (+ bias[e]), fp32 accumulation.
// One warp per (expert, token); lane covers d = 8*lane + 256*i.
template <typename TX, typename TW>
__global__ void __launch_bounds__(256) router_logits_kernel(const TX *__restrict__ x,
                                                            const TW *__restrict__ wr,
                                                            const float *__restrict__ bias,
                                                            int64_t T, int D, int E, int tb,
                                                            float *__restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= E) return;
  const int64_t t0 = (int64_t)blockIdx.y * tb;
  const int64_t t1 = min(T, t0 + tb);
  const TW *row = wr + (int64_t)e * D;
  const float b = bias ? bias[e] : 0.0f;
  for (int64_t t = t0; t < t1; ++t) {
    const TX *xr = x + t * D;
    float acc = 0.0f;
    for (int d = 8 * lane; d < D; d += 256) {
      float wv[8], xv[8];
      load8<TW>(row + d, wv);
      load8<TX>(xr + d, xv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(xv[i], wv[i], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) logits[t * E + e] = acc + b;
  }
}

// Small batches (T <= 64, D a multiple of 1024): two experts per block and a
// quarter of n_embd per warp.  The warp keeps its quarter of the router row
// in registers (NCH 8-element chunks per lane) and walks the tokens in
// batches of 16 / NCH, all of a batch's loads issued before any use; the
// quarters are added in a fixed order.
template <typename TX, typename TW, int NCH>
__global__ void __launch_bounds__(256) router_small_kernel(const TX *__restrict__ x,
                                                           const TW *__restrict__ wr,
                                                           const float *__restrict__ bias, int T,
                                                           int D, int E, float *__restrict__ logits) {
  // a kernel launched after this one with programmatic dependent launch may
  // start its independent work now (it waits for this grid before reading
  // the logits)
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int TB = 16 / NCH;  // tokens per batch
  __shared__ float part[8][64];  // [warp][token] partial logits
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 2 + (warp >> 2), c0 = (warp & 3) * (D / 4);
  if (e < E) {
    float wv[NCH][8];
#pragma unroll
    for (int c = 0; c < NCH; ++c) load8<TW>(wr + (int64_t)e * D + c0 + 256 * c + 8 * lane, wv[c]);
    for (int t0 = 0; t0 < T; t0 += TB) {
      float xv[TB][NCH][8];
#pragma unroll
      for (int u = 0; u < TB; ++u)
        if (t0 + u < T) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) load8<TX>(x + (int64_t)(t0 + u) * D + c0 + 256 * c + 8 * lane, xv[u][c]);
        }
      float acc[TB];
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        acc[u] = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[u] = fmaf(xv[u][c][i], wv[c][i], acc[u]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < TB; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < TB; ++u)
          if (t0 + u < T) part[warp][t0 + u] = acc[u];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * T; i += blockDim.x) {
    const int r = i / T, t = i % T, ee = blockIdx.x * 2 + r;
    if (ee < E)
      logits[(int64_t)t * E + ee] =
          ((part[4 * r][t] + part[4 * r + 1][t]) + part[4 * r + 2][t]) + part[4 * r + 3][t] + (bias ? bias[ee] : 0.f);
  }
}

template <typename TX, typename TW>
cudaError_t launch_router_small(const TX *x, const TW *wr, const float *bias, int T, int D, int E, float *logits,
                                cudaStream_t s) {
  const dim3 g((E + 1) / 2);
  switch (D / 1024) {  // 8-element chunks per lane: D / 4 / 256
    case 1: router_small_kernel<TX, TW, 1><<<g, 256, 0, s>>>(x, wr, bias, T, D, E, logits); break;
    case 2: router_small_kernel<TX, TW, 2><<<g, 256, 0, s>>>(x, wr, bias, T, D, E, logits); break;
    case 4: router_small_kernel<TX, TW, 4><<<g, 256, 0, s>>>(x, wr, bias, T, D, E, logits); break;
    case 8: router_small_kernel<TX, TW, 8><<<g, 256, 0, s>>>(x, wr, bias, T, D, E, logits); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) select_kernel(const float *__restrict__ logits, int64_t T,
                                                     int E, int k, float routed_scale, float logit_scale,
                                                     const float *__restrict__ unbias, int32_t *__restrict__ ids,
                                                     float *__restrict__ w, unsigned *st) {
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  select_token(logits + t * E, E, k, routed_scale, logit_scale, unbias, ids + t * k, w + t * k, st);
}

// Stable rank of each pair of one chunk inside its expert, in ascending pair
// order: the rank within the warp from a match mask, plus the counts of the
// same expert in the chunk's earlier warps.  Block = ROUTE_CHUNK threads.
// wtab: [32][E] shared counters.
__device__ int chunk_rank(int e, bool valid, int *wtab, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wtab[i] = 0;
  __syncthreads();
  const unsigned act = __ballot_sync(0xffffffffu, valid);
  const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1) & act;
  const int in_warp = __popc(same & ((1u << lane) - 1u));
  if (valid && in_warp == 0) wtab[warp * E + e] = __popc(same);
  __syncthreads();
  int r = in_warp;
  if (valid)
    for (int w2 = 0; w2 < warp; ++w2) r += wtab[w2 * E + e];
  return r;
}

// Small batches (T*k <= ROUTE_CHUNK): selection for every token, histogram,
// exclusive scan, stable permutation and used-expert list, all in one block.
__global__ void __launch_bounds__(ROUTE_CHUNK) select_route_small_kernel(
    const float *__restrict__ logits, int64_t T, int E, int k, float routed_scale, float logit_scale,
    const float *__restrict__ unbias, int32_t *__restrict__ ids, float *__restrict__ w, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ pos,
    int32_t *__restrict__ used, unsigned *st) {
  extern __shared__ int sm[];
  int *cnt = sm;           // [E]
  int *off = cnt + E;      // [E+1]
  int *wtab = off + E + 1; // [32][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t t = warp; t < T; t += blockDim.x / 32)
    select_token(logits + t * E, E, k, routed_scale, logit_scale, unbias, ids + t * k, w + t * k, st);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t P = T * k;
  const int p = threadIdx.x;
  const bool valid = p < P;
  int e = valid ? ids[p] : 0;
  if (valid && (e < 0 || e >= E)) { flag(st, ST_BAD_ID); e = 0; }
  if (valid) atomicAdd(&cnt[e], 1);
  __syncthreads();
  if (warp == 0) {  // exclusive scan of counts and the used-expert list
    int run = 0, nu = 0;
    for (int base = 0; base < E; base += 32) {
      int c = base + lane < E ? cnt[base + lane] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (base + lane < E) {
        off[base + lane] = run + incl - c;
        counts[base + lane] = c;
        offsets[base + lane] = run + incl - c;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      unsigned m = __ballot_sync(0xffffffffu, c > 0);
      if (c > 0) used[nu + __popc(m & ((1u << lane) - 1u))] = base + lane;
      nu += __popc(m);
    }
    if (lane == 0) { off[E] = run; offsets[E] = run; used[E] = nu; }
  }
  __syncthreads();
  const int r = chunk_rank(e, valid, wtab, E);
  if (valid) {
    const int at = off[e] + r;
    perm[at] = p;
    pos[p] = at;
  }
}

// Large batches: per-chunk histograms ...
__global__ void __launch_bounds__(ROUTE_CHUNK) route_hist_kernel(const int32_t *__restrict__ ids,
                                                                 int64_t P, int E,
                                                                 int32_t *__restrict__ chunk,
                                                                 unsigned *st) {
  extern __shared__ int h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * ROUTE_CHUNK + threadIdx.x;
  if (p < P) {
    int e = ids[p];
    if (e < 0 || e >= E) { flag(st, ST_BAD_ID); e = 0; }
    atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk[(int64_t)blockIdx.x * E + e] = h[e];
}

// ... one block turns them into counts, offsets, per-chunk bases and the
// used-expert list ...
__global__ void __launch_bounds__(1024) route_scan_kernel(int32_t *__restrict__ chunk,
                                                          int64_t n_chunks, int E,
                                                          int32_t *__restrict__ counts,
                                                          int32_t *__restrict__ offsets,
                                                          int32_t *__restrict__ used) {
  __shared__ int tot[1024];
  __shared__ int warp_sums[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int run = 0;
  if (e < E)
    for (int64_t c = 0; c < n_chunks; ++c) {
      int v = chunk[c * E + e];
      chunk[c * E + e] = run;
      run += v;
    }
  tot[e] = e < E ? run : 0;
  // block-wide exclusive scan of tot
  int incl = tot[e];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += v;
    }
    warp_sums[lane] = si - s;
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - tot[e];
  if (e < E) {
    counts[e] = tot[e];
    offsets[e] = excl;
    for (int64_t c = 0; c < n_chunks; ++c) chunk[c * E + e] += excl;
  }
  if (e == E - 1) offsets[E] = excl + tot[e];
  __syncthreads();
  // used-expert list (ascending): rank = number of earlier experts with tokens
  const bool has = e < E && tot[e] > 0;
  const unsigned m = __ballot_sync(0xffffffffu, has);
  __shared__ int wcnt[32];
  if (lane == 0) wcnt[warp] = __popc(m);
  __syncthreads();
  int before = 0;
  for (int w2 = 0; w2 < warp; ++w2) before += wcnt[w2];
  if (has) used[before + __popc(m & ((1u << lane) - 1u))] = e;
  if (e == 0) {
    int n = 0;
    for (int w2 = 0; w2 < 32; ++w2) n += wcnt[w2];
    used[E] = n;
  }
}

// ... and every chunk scatters its pairs to their stable positions.
__global__ void __launch_bounds__(ROUTE_CHUNK) route_scatter_kernel(
    const int32_t *__restrict__ ids, int64_t P, int E, const int32_t *__restrict__ chunk,
    int32_t *__restrict__ perm, int32_t *__restrict__ pos) {
  extern __shared__ int wtab[];
  const int64_t p = (int64_t)blockIdx.x * ROUTE_CHUNK + threadIdx.x;
  const bool valid = p < P;
  int e = valid ? ids[p] : 0;
  if (e < 0 || e >= E) e = 0;
  const int r = chunk_rank(e, valid, wtab, E);
  if (valid) {
    const int at = chunk[(int64_t)blockIdx.x * E + e] + r;
    perm[at] = (int32_t)p;
    pos[p] = at;
  }
}

}  // namespace

cudaError_t launch_route(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                         cudaStream_t s) {
  cudaError_t err = launch_router_logits(sh, W, x, wk, s);
  if (err != cudaSuccess) return err;
  return launch_select_route(sh, wk, W.router_bias, s);
}

cudaError_t launch_router_logits(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                                 cudaStream_t s) {
  const int64_t T = wk.T;
  const int E = sh.E, D = sh.D;
  unsigned *st = status_word();
  const int tb = T <= 64 ? (int)T : 16;
  dim3 g((E + 7) / 8, (unsigned)((T + tb - 1) / tb));
  const int dq = D / 1024;
  if (T <= 64 && D % 1024 == 0 && (dq == 1 || dq == 2 || dq == 4 || dq == 8) && sh.x_dtype == sh.router_dtype) {
    cudaError_t e2 = sh.x_dtype == DS_BF16
                         ? launch_router_small<uint16_t, uint16_t>((const uint16_t *)x, (const uint16_t *)W.router_w,
                                                                   W.router_bias, (int)T, D, E, wk.logits, s)
                         : launch_router_small<float, float>((const float *)x, (const float *)W.router_w,
                                                             W.router_bias, (int)T, D, E, wk.logits, s);
    if (e2 != cudaSuccess) return e2;
  } else if (sh.x_dtype == DS_BF16) {
    if (sh.router_dtype == DS_BF16)
      router_logits_kernel<uint16_t, uint16_t><<<g, 256, 0, s>>>(
          (const uint16_t *)x, (const uint16_t *)W.router_w, W.router_bias, T, D, E, tb, wk.logits);
    else
      router_logits_kernel<uint16_t, float><<<g, 256, 0, s>>>(
          (const uint16_t *)x, (const float *)W.router_w, W.router_bias, T, D, E, tb, wk.logits);
  } else {
    if (sh.router_dtype == DS_BF16)
      router_logits_kernel<float, uint16_t><<<g, 256, 0, s>>>(
          (const float *)x, (const uint16_t *)W.router_w, W.router_bias, T, D, E, tb, wk.logits);
    else
      router_logits_kernel<float, float><<<g, 256, 0, s>>>(
          (const float *)x, (const float *)W.router_w, W.router_bias, T, D, E, tb, wk.logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_select_route(const Shape &sh, const Work &wk, const float *bias, cudaStream_t s) {
  const float *unbias = sh.bias_select_only ? bias : nullptr;
  const int64_t T = wk.T;
  const int E = sh.E, k = sh.k;
  unsigned *st = status_word();
  const int64_t P = T * k;
  cudaError_t err;
  static OncePerDevice once;
  err = once_per_device(once, []() {  // up to 33E+1 ints (E <= 1024: 132 KB) of dynamic shared memory
    cudaError_t e = cudaFuncSetAttribute(select_route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         140 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 140 * 1024);
    return e;
  });
  if (err != cudaSuccess) return err;
  if (P <= ROUTE_CHUNK) {
    size_t smem = sizeof(int) * (size_t)(E + E + 1 + 32 * E);
    select_route_small_kernel<<<1, ROUTE_CHUNK, smem, s>>>(wk.logits, T, E, k, sh.routed_scale, sh.logit_scale, unbias,
                                                           wk.ids, wk.w, wk.counts, wk.offsets,
                                                           wk.perm, wk.pos, wk.used, st);
    return cudaGetLastError();
  }
  select_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(wk.logits, T, E, k, sh.routed_scale, sh.logit_scale, unbias, wk.ids,
                                                        wk.w, st);
  const int64_t nc = (P + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
  route_hist_kernel<<<(unsigned)nc, ROUTE_CHUNK, sizeof(int) * E, s>>>(wk.ids, P, E, wk.chunk, st);
  route_scan_kernel<<<1, 1024, 0, s>>>(wk.chunk, nc, E, wk.counts, wk.offsets, wk.used);
  route_scatter_kernel<<<(unsigned)nc, ROUTE_CHUNK, sizeof(int) * 32 * E, s>>>(wk.ids, P, E,
                                                                              wk.chunk, wk.perm,
                                                                              wk.pos);
  return cudaGetLastError();
}

}  // namespace dsm
