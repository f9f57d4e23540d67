// Decode path for a few tokens (T*k <= 32, e.g. one token at 4096/256/6/2048):
// three kernels chained with programmatic dependent launch (PDL).
//
// What it computes is the layer of "Understanding Dwarf Star" 5.3.2/5.3.7
// (router -> top-k -> gate/up -> SiLU(gate)*up -> down -> weighted sum, plus
// the always-active shared expert of 5.3.4), with the routed weights read as
// Q2_K blocks (3.3.3) and dequantised on the fly (2.8.1-2.8.2).
//
//   K1 route_kernel   router logits (a quarter of a row per warp).
//   K2 gateup_kernel  one warp per CTA waits for K1 and selects the top-k and
//                     builds the route (each CTA its own copy; CTA 0 publishes
//                     it), while the other warps start on the shared gate/up
//                     quarter-rows (no route needed: they overlap K1 through
//                     PDL); then one warp per routed gate/up row pair ->
//                     h = SiLU(g) * u.
//   K3 down_kernel    one warp per output row: shared down row, every used
//                     expert's down row, and the combine
//                     out = y_shared + sum_j w_j y_j (slot order j).
//
// Q2_K rows are read straight from global memory (every byte once; a lane's
// 4-byte words of one 84-byte block), all loads of an item issued before any
// use.  Dot products with Q2_K rows are exact integer sums: activations are
// turned into 16-bit fixed point per 256-element block, X = rint(v / step),
// step = 2^(e-15) with max |v| < 2^e, split in a signed high byte and an
// unsigned low byte, and sum_j q_j X_j is formed with dp4a; per lane the
// integers sum_s sc_s S_s and sum_s m_s sum(X) are accumulated exactly and
// converted once: w.x = step * (d * sum sc S - dmin * sum m X).  The only
// rounding beyond fp32 is that fixed point (|err| <= 2^-16 of the block's
// largest |v| per element).
//
// Q4_K rows ("Understanding Dwarf Star", 2.3.2: 144-byte blocks, 8
// sub-blocks of 32 with 6-bit scales and mins, 4-bit codes) use the same
// scheme with their own lane map and planes (the even and odd nibbles of each
// code word); every kernel here is a template over the row format (Q2Rows /
// Q4Rows, defined with the streaming kernel).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "qrows.cuh"
#include "select.cuh"

namespace dsm {
namespace {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // bound of every wait

#ifdef DS_MOE_TEST_HOOKS
// Test build only (never in the library the product loads): bit 0 of
// g_test_hook_flags keeps the route from being published to the block, so
// that every wait for it runs out, and a nonzero g_test_hook_limit_ns
// replaces the bound of the waits for the route, the ring stages and the grid
// barrier (the final wait for a block's own copies keeps the full bound).
__device__ unsigned g_test_hook_flags;
__device__ unsigned long long g_test_hook_limit_ns;
__device__ __forceinline__ uint64_t wait_limit() {
  return g_test_hook_limit_ns ? (uint64_t)g_test_hook_limit_ns : WAIT_LIMIT_NS;
}
__device__ __forceinline__ bool hold_route() { return (g_test_hook_flags & 1u) != 0; }
#else
__device__ __forceinline__ uint64_t wait_limit() { return WAIT_LIMIT_NS; }
__device__ __forceinline__ bool hold_route() { return false; }
#endif

constexpr int PMAXD = 32;          // token-expert pairs this path serves (one per lane)
constexpr int NW2 = 12, NW3 = 12;  // warps per CTA of K2 and K3
constexpr size_t SMEM_LIMIT = 227 * 1024;

enum {
  C_NUSED = 1,  // control word: experts with tokens (written with the route)
  C_BAR = 2,    // control word: grid barrier of the one-token streaming kernel
};


struct Args {
  int D, E, F, Fs, k, T;
  float routed_scale, logit_scale;
  int bias_select_only;  // the router bias steers the selection only
  const void *router_w;
  int router_f32;
  const float *bias;
  const uint16_t *sg, *su, *sd;
  const uint8_t *experts;
  int64_t expert_bytes, gate_bytes;
  // expert residency (null slot: every expert at experts + e * expert_bytes)
  const int32_t *slot;   // [E]: cache slot of expert e, or -1: read it from host
  const uint8_t *cache;  // device slots of expert_bytes each
  const uint8_t *host;   // device view of the host copy of all E experts
  const void *x;
  int x_f32;
  void *x_stage;  // non-null: x is host memory; the router grid copies it here for the streaming kernel
  float *logits;
  int32_t *ids;
  float *w;
  int32_t *counts, *offsets, *perm, *pos, *used;
  float *h;    // [P][F] routed activations, perm order
  float *hs;   // [T][Fs] shared-expert activations (streaming kernel)
  float *pgu;  // [2][4][T][Fs] shared gate / up partial sums (per quarter of n_embd)
  unsigned *ctrl;
  float *out;
  int accumulate;
  unsigned *status;
  int n_slots;
};

// Packed bytes of expert e: its cache slot when it has one, else the host
// copy (far = true: read with ordinary loads, never with bulk copies); without
// a slot table the experts array.  The same bytes either way.
__device__ __forceinline__ const uint8_t *expert_at(const Args &a, int e, bool &far) {
  if (!a.slot) {
    far = false;
    return a.experts + (int64_t)e * a.expert_bytes;
  }
  const int s = __ldg(a.slot + e);
  far = s < 0;
  return far ? a.host + (int64_t)e * a.expert_bytes : a.cache + (int64_t)s * a.expert_bytes;
}

template <typename T>
__device__ __forceinline__ void ld8(const T *p, float v[8]);
template <>
__device__ __forceinline__ void ld8<float>(const float *p, float v[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void ld8<uint16_t>(const uint16_t *p, float v[8]) {
  bf16x8(__ldg(reinterpret_cast<const uint4 *>(p)), v);
}

// ===================================================================== K1 ==

// Router logits: two expert rows per CTA, a quarter of n_embd per warp (at
// most 32 registers per thread, so that the CTA fits beside a streaming CTA).
template <typename TX, typename TW>
__global__ void __launch_bounds__(256, 8) route_kernel(const Args a) {
  // This grid may be launched while the previous kernel of the stream (the
  // streaming kernel of the previous layer) still runs: its router rows do
  // not depend on it and are started towards L2 at once; x and the workspace
  // are touched only after that grid has completed.
  if (threadIdx.x == 0 && 2 * blockIdx.x < a.E) {
    const int rows = min(2, a.E - 2 * (int)blockIdx.x);
    bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(a.router_w) + (int64_t)2 * blockIdx.x * a.D * sizeof(TW),
                     (uint32_t)(rows * a.D * sizeof(TW)));
  }
  pdl_wait();
  pdl_trigger();  // the next kernel may start its route-free work now
  // The dependent kernel touches this word only after its griddepcontrol.wait,
  // i.e. after this grid has completed.
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ctrl[C_BAR] = 0u;
  if (a.x_stage && blockIdx.x == 0) {  // one device copy of x for the next kernel
    const size_t n16 = (size_t)a.T * a.D * (a.x_f32 ? 4 : 2) / 16;
    for (size_t i = threadIdx.x; i < n16; i += blockDim.x)
      reinterpret_cast<uint4 *>(a.x_stage)[i] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
  }
  __shared__ float part[8][4];  // [warp][token] partial logits
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // two expert rows per CTA, a quarter of n_embd per warp, loads issued up front
  const int e = blockIdx.x * 2 + (warp >> 2), qd = warp & 3, len = a.D / 4, c0 = qd * len;
  if (e < a.E) {
    const TW *row = (const TW *)a.router_w + (int64_t)e * a.D + c0;
    for (int t = 0; t < a.T; ++t) {
      const TX *xr = (const TX *)a.x + (int64_t)t * a.D + c0;
      float acc = 0.f;
#pragma unroll 4
      for (int d = 8 * lane; d < len; d += 256) {
        float wv[8], xv[8];
        ld8<TW>(row + d, wv);
        ld8<TX>(xr + d, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(xv[i], wv[i], acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) part[warp][t] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * a.T) {
    const int r = threadIdx.x / a.T, t = threadIdx.x % a.T, ee = blockIdx.x * 2 + r;
    if (ee < a.E) {
      const float v = ((part[4 * r][t] + part[4 * r + 1][t]) + part[4 * r + 2][t]) + part[4 * r + 3][t];
      a.logits[(int64_t)t * a.E + ee] = v + (a.bias ? a.bias[ee] : 0.f);
    }
  }
}

// The route as the warps of K2/K3 keep it in registers: lane p holds pair p,
// lane u holds used expert u.
struct RouteCache {
  int nu, perm, used, base, cnt;
  float w;
  int pos;  // lane p: position of pair p in the route (select_route_warp only)
};

// Selection and route by one warp (T * k <= 32): top-k by logit, ties to the
// lower index, weights = routed_scale * softmax over logit_scale * the selected logits; the
// stable route puts pair p at #(pairs with a smaller expert, or the same
// expert and a smaller p).  Returns the calling lane's RouteCache entries; with
// publish, also writes ids, w, counts, offsets, perm, pos and used.
template <int PMAX>
__device__ RouteCache select_route_warp(const Args &a, bool publish) {
  const int lane = threadIdx.x & 31, P = a.T * a.k;
  int my_id = 0;     // lane p: expert of pair p
  float my_lg = 0.f; // lane p: its logit
  const int nv = (a.E + 31) / 32;  // logits per lane (E <= 1024)
  for (int t = 0; t < a.T; ++t) {
    const float *L = a.logits + (int64_t)t * a.E;
    float lv[32];
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) lv[ii] = ii < nv && lane + 32 * ii < a.E ? __ldcg(L + lane + 32 * ii) : -INFINITY;
    if (a.E <= 256) {  // eight candidates per lane, sorted once
      topk_sorted8(lv, a.E, a.k, my_id, my_lg, a.status, t * a.k);
      continue;
    }
    // each lane's best remaining candidate (largest logit, then lowest
    // index); per pick the warp takes the best of those, and only the lane
    // that supplied it looks for its next one
    uint32_t taken = 0;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    auto rescan = [&]() {
      bv = -INFINITY;
      bi = 0x7fffffff;
#pragma unroll
      for (int ii = 0; ii < 32; ++ii) {
        if (ii >= nv) break;
        const int ee = lane + 32 * ii;
        if (ee < a.E && !(taken & (1u << ii)) && (lv[ii] > bv || (lv[ii] == bv && ee < bi))) { bv = lv[ii]; bi = ee; }
      }
    };
    rescan();
    for (int j = 0; j < a.k; ++j) {
      // the warp's largest logit (as an order-preserving unsigned key, two
      // hardware reductions), then the lowest index holding it
      const uint32_t key = ord_key(bv + 0.f);  // -0 as +0: equal logits tie
      const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
      int wi = (int)__reduce_min_sync(0xffffffffu, key == mk ? (uint32_t)bi : 0x7fffffffu);
      const float wv = ord_val(mk);
      if (wi < 0 || wi >= a.E) { if (lane == 0 && publish) flag(a.status, ST_BAD_ID); wi = 0; }
      if ((wi & 31) == lane && wi == bi) {
        taken |= 1u << (wi >> 5);
        rescan();
      }
      if (lane == t * a.k + j) { my_id = wi; my_lg = wv; }
    }
  }
  // weights: softmax over each token's selected logits
  const int tok = lane / max(a.k, 1), j0 = tok * a.k;
  // (with the bias steering the selection only, it is taken back out here)
  const float my_u = a.bias_select_only && a.bias && lane < P ? my_lg - __ldg(a.bias + my_id) : my_lg;
  const float m0 = __shfl_sync(0xffffffffu, my_u, min(j0, 31));
  float ex = lane < P ? __expf(a.logit_scale * (my_u - m0)) : 0.f;
  // every pair's expert, exponential and (below) rank in registers: the
  // shuffles are independent and issue back to back
  int idq[PMAX];  // (PMAX >= T * k)
#pragma unroll
  for (int q = 0; q < PMAX; ++q) idq[q] = __shfl_sync(0xffffffffu, my_id, q);
  float exj[PMAX];  // the exponentials of this lane's token, pick order
#pragma unroll
  for (int j = 0; j < PMAX; ++j) exj[j] = __shfl_sync(0xffffffffu, ex, min(j0 + j, 31));
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < PMAX; ++j)
    if (j < a.k) den += exj[j];
  const float my_w = lane < P ? a.routed_scale * (ex / den) : 0.f;
  // ranks
  int rank = 0, first = 1, ui = 0;
#pragma unroll
  for (int q = 0; q < PMAX; ++q)
    if (q < P) {
      rank += (idq[q] < my_id) || (idq[q] == my_id && q < lane);
      if (idq[q] == my_id && q < lane) first = 0;
    }
  const unsigned firsts = __ballot_sync(0xffffffffu, lane < P && first);
#pragma unroll
  for (int q = 0; q < PMAX; ++q)  // distinct experts below mine
    if (q < P) ui += ((firsts >> q) & 1u) && idq[q] < my_id;
  RouteCache r;
  r.nu = __popc(firsts);
  int rkq[PMAX], uiq[PMAX];
#pragma unroll
  for (int q = 0; q < PMAX; ++q) {
    rkq[q] = __shfl_sync(0xffffffffu, rank, q);
    uiq[q] = __shfl_sync(0xffffffffu, ui, q);
  }
  // lane p learns perm[p]: the pair whose rank is p
  int perm_p = 0;
#pragma unroll
  for (int q = 0; q < PMAX; ++q)
    if (q < P && rkq[q] == lane) perm_p = q;
  r.perm = perm_p;
  r.w = my_w;
  r.pos = rank;
  // lane u learns used[u], its first position and its pair count
  int used_u = 0, base_u = 0, cnt_u = 0;
#pragma unroll
  for (int q = 0; q < PMAX; ++q)
    if (q < P && ((firsts >> q) & 1u) && uiq[q] == lane) { used_u = idq[q]; base_u = rkq[q]; }
#pragma unroll
  for (int q = 0; q < PMAX; ++q)
    if (q < P) cnt_u += (lane < r.nu && idq[q] == used_u) ? 1 : 0;
  r.used = used_u;
  r.base = base_u;
  r.cnt = cnt_u;
  if (publish) {
    if (lane < P) {
      a.ids[lane] = my_id;
      a.w[lane] = my_w;
      a.perm[rank] = lane;
      a.pos[lane] = rank;
    }
    if (lane < r.nu) a.used[lane] = used_u;
    for (int e0 = 0; e0 <= a.E; e0 += 32) {  // warp-uniform trip count (shuffles inside)
      const int e = e0 + lane;
      int lt = 0, eqc = 0;
      for (int q = 0; q < P; ++q) {
        const int eq = __shfl_sync(0xffffffffu, my_id, q);
        lt += eq < e;
        eqc += eq == e;
      }
      if (e <= a.E) a.offsets[e] = lt;
      if (e < a.E) a.counts[e] = eqc;
    }
    if (lane == 0) {
      a.used[a.E] = r.nu;
      a.ctrl[C_NUSED] = (unsigned)r.nu;
    }
  }
  return r;
}

// Reads the route published in global memory; any entry out of range (which
// a correct route never has) is replaced by a harmless value and flagged.
__device__ __forceinline__ RouteCache load_route(const Args &a) {
  const int lane = threadIdx.x & 31, P = a.T * a.k;
  RouteCache r;
  r.pos = 0;
  r.nu = (int)__ldcg((const int *)(a.ctrl + C_NUSED));
  bool bad = r.nu < 0 || r.nu > P;
  if (bad) r.nu = 0;
  r.perm = lane < P ? __ldcg(a.perm + lane) : 0;
  r.w = lane < P ? __ldcg(a.w + lane) : 0.f;
  r.used = lane < r.nu ? __ldcg(a.used + lane) : 0;
  if (r.used < 0 || r.used >= a.E) { bad = true; r.used = 0; }
  r.base = lane < r.nu ? __ldcg(a.offsets + r.used) : 0;
  r.cnt = lane < r.nu ? __ldcg(a.offsets + r.used + 1) - r.base : 0;
  if (r.perm < 0 || r.perm >= P || r.base < 0 || r.cnt < 0 || r.base + r.cnt > P) {
    bad = true;
    r.perm = 0; r.base = 0; r.cnt = 0;
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) flag(a.status, ST_BAD_COUNT);
    r.nu = 0;  // compute nothing routed rather than index with bad data
  }
  return r;
}

// ===================================================================== K2 ==

// R: the row format of the n_embd-long rows (Q2Rows / Q4Rows, defined with
// the streaming kernel below; a template, so resolved at instantiation).
template <class R>
__global__ void __launch_bounds__(NW2 * 32, 1) gateup_kernel(const Args a) {
  pdl_trigger();  // every CTA of this grid is resident: the down kernel may queue
  extern __shared__ __align__(16) uint32_t xpl[];  // [T] planes + steps
  __shared__ int s_rt[5][32];
  __shared__ float s_w[32];
  __shared__ volatile int s_ready;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = a.D / QK, nsb = a.D / R::SUB, xw = R::NPL * nsb + nb;
  if (threadIdx.x == 0) s_ready = 0;
  for (int u = warp; u < (a.T * nb + 1) / 2; u += NW2) {
    const int bi = min(2 * u + (lane >> 4), a.T * nb - 1);
    const int t = bi / nb, b = bi % nb;
    const int64_t e0 = (int64_t)t * a.D + QK * b + 16 * (lane & 15);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = a.x_f32 ? __ldg((const float *)a.x + e0 + j) : bf16_to_f32(__ldg((const uint16_t *)a.x + e0 + j));
    R::digitize(v, b, xpl + t * xw, reinterpret_cast<float *>(xpl + t * xw + R::NPL * nsb), nsb);
  }
  __syncthreads();
  if (warp == 0) {
    // every CTA selects and routes on its own (a few hundred logits); CTA 0
    // also publishes the route for the down kernel and the debug outputs
    pdl_wait();  // the router logits are complete and visible
    const RouteCache r = select_route_warp<PMAXD>(a, blockIdx.x == 0);
    s_rt[0][lane] = r.perm; s_rt[1][lane] = r.used; s_rt[2][lane] = r.base; s_rt[3][lane] = r.cnt;
    s_rt[4][lane] = r.nu;
    s_w[lane] = r.w;
    __threadfence_block();
    __syncwarp();
    if (lane == 0 && !hold_route()) s_ready = 1;
  }

  const int n_sh = a.Fs > 0 ? 4 * a.Fs : 0;    // shared items: (row, quarter of n_embd)
  const int n_items = n_sh + a.n_slots * a.F;  // then one per routed (slot, row)
  const int gw = warp * gridDim.x + blockIdx.x, nwork = gridDim.x * NW2;
  const int rb = nb * R::BB;
  bool have_route = false;
  RouteCache rc{0, 0, 0, 0, 0, 0.f, 0};
  // L2 prefetch (bulk-copy engine, lane 0) of item i's bytes; every lane calls
  // it (the routed address comes from a shuffle)
  auto prefetch = [&](int i) {
    if (i >= n_items) return;
    if (i < n_sh) {
      if (lane == 0) {
        const int f = i >> 2, q = i & 3, len = a.D / 4;
        bulk_prefetch_l2(a.sg + (int64_t)f * a.D + q * len, (uint32_t)len * 2u);
        bulk_prefetch_l2(a.su + (int64_t)f * a.D + q * len, (uint32_t)len * 2u);
      }
    } else if (have_route) {
      const int r = i - n_sh, slot = r / a.F, f = r % a.F;
      const int e = shfl(rc.used, min(slot, 31));
      if (slot < rc.nu && lane == 0) {
        bool far;
        const uint8_t *g = expert_at(a, e, far) + (int64_t)f * rb;
        if (!far) {
          bulk_prefetch_l2(g, (uint32_t)rb);
          bulk_prefetch_l2(g + a.gate_bytes, (uint32_t)rb);
        }
      }
    }
  };
  prefetch(gw);
  prefetch(gw + nwork);
  for (int it = gw; it < n_items; it += nwork) {
    if (it >= n_sh && !have_route) {
      int ok = 1;
      if (lane == 0) {  // bounded wait for this CTA's route
        const uint64_t t0 = globaltimer_ns();
        while (!s_ready) {
          if (globaltimer_ns() - t0 > wait_limit()) { flag(a.status, ST_TIMEOUT); ok = 0; break; }
          __nanosleep(64);
        }
      }
      if (!shfl(ok, 0)) return;
      __syncwarp();
      rc.perm = s_rt[0][lane]; rc.used = s_rt[1][lane]; rc.base = s_rt[2][lane]; rc.cnt = s_rt[3][lane];
      rc.nu = s_rt[4][lane]; rc.w = s_w[lane];
      have_route = true;
      prefetch(it + nwork);  // routed items could not be prefetched before
    }
    prefetch(it + 2 * nwork);
    if (it < n_sh) {
      const int f = it >> 2, q = it & 3, len = a.D / 4, c0 = q * len;
      const uint16_t *gr = a.sg + (int64_t)f * a.D + c0, *ur = a.su + (int64_t)f * a.D + c0;
      float gu[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // gate[0..3], up[0..3] (T <= 4)
#pragma unroll 4
      for (int c = 8 * lane; c < len; c += 256) {
        float gf[8], uf[8];
        bf16x8(__ldcs(reinterpret_cast<const uint4 *>(gr + c)), gf);
        bf16x8(__ldcs(reinterpret_cast<const uint4 *>(ur + c)), uf);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (t >= a.T) break;
          float xf[8];
          if (a.x_f32) ld8<float>((const float *)a.x + (int64_t)t * a.D + c0 + c, xf);
          else ld8<uint16_t>((const uint16_t *)a.x + (int64_t)t * a.D + c0 + c, xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) { gu[t] = fmaf(gf[i], xf[i], gu[t]); gu[4 + t] = fmaf(uf[i], xf[i], gu[4 + t]); }
        }
      }
      warp_sum_n<8>(gu);
      if (lane < 2 * a.T) {  // lane = matrix * T + token
        const int m = lane / a.T, t = lane % a.T;
        a.pgu[((int64_t)(m * 4 + q) * a.T + t) * a.Fs + f] = gu[4 * m + t];
      }
      continue;
    }
    const int r = it - n_sh, slot = r / a.F, f = r % a.F;
    if (slot >= rc.nu) continue;
    const int e = shfl(rc.used, slot), base = shfl(rc.base, slot), n = shfl(rc.cnt, slot);
    bool far;
    const uint8_t *grow = expert_at(a, e, far) + (int64_t)f * rb;
    typename R::Row gp, up;
    R::load_g(grow, gp);
    R::load_g(grow + a.gate_bytes, up);
    for (int j = 0; j < n; ++j) {
      const int t = shfl(rc.perm, base + j) / a.k;
      const uint32_t *pl = xpl + t * xw;
      const float *st = reinterpret_cast<const float *>(pl + R::NPL * nsb);
      float gu[2] = {R::dot(gp, pl, st, nsb), R::dot(up, pl, st, nsb)};
      warp_sum_n<2>(gu);
      if (lane == 0) a.h[(int64_t)(base + j) * a.F + f] = silu(gu[0]) * gu[1];
    }
  }
}

// ===================================================================== K3 ==

// R: the row format of the n_ff-long rows.
template <class R>
__global__ void __launch_bounds__(NW3 * 32, 1) down_kernel(const Args a) {
  pdl_wait();  // gate/up (and through it the route) complete and visible
  extern __shared__ __align__(16) uint32_t hpl[];  // [P] planes + steps, then hs [T][Fs]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = a.F / QK, nsb = a.F / R::SUB, hw = R::NPL * nsb + nb;
  const int P = a.T * a.k;
  float *hs = reinterpret_cast<float *>(hpl + P * hw);
  const RouteCache rc = load_route(a);
  // h of every pair in fixed point (perm order), and the shared activations
  for (int u = warp; u < (P * nb + 1) / 2; u += NW3) {
    const int bi = min(2 * u + (lane >> 4), P * nb - 1);
    const int q = bi / nb, b = bi % nb;
    const float4 *src = reinterpret_cast<const float4 *>(a.h + (int64_t)q * a.F + QK * b + 16 * (lane & 15));
    float v[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 f4 = __ldcg(src + j);
      v[4 * j] = f4.x; v[4 * j + 1] = f4.y; v[4 * j + 2] = f4.z; v[4 * j + 3] = f4.w;
    }
    R::digitize(v, b, hpl + q * hw, reinterpret_cast<float *>(hpl + q * hw + R::NPL * nsb), nsb);
  }
  {
    // shared activations: hs = SiLU(sum of gate quarters) * (sum of up quarters),
    // quarters summed in a fixed order; all loads of a thread issued first
    constexpr int PER = 8;  // elements per thread and pass
    for (int i0 = threadIdx.x; i0 < a.T * a.Fs; i0 += PER * blockDim.x) {
      float g[PER][4], u[PER][4];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i = i0 + k * blockDim.x;
        const int t = i / max(a.Fs, 1), f = i % max(a.Fs, 1);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          g[k][q] = i < a.T * a.Fs ? __ldcg(a.pgu + ((int64_t)(0 * 4 + q) * a.T + t) * a.Fs + f) : 0.f;
          u[k][q] = i < a.T * a.Fs ? __ldcg(a.pgu + ((int64_t)(1 * 4 + q) * a.T + t) * a.Fs + f) : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i = i0 + k * blockDim.x;
        if (i < a.T * a.Fs)
          hs[i] = silu(((g[k][0] + g[k][1]) + g[k][2]) + g[k][3]) * (((u[k][0] + u[k][1]) + u[k][2]) + u[k][3]);
      }
    }
  }
  __syncthreads();

  const int gw = warp * gridDim.x + blockIdx.x, nwork = gridDim.x * NW3;
  const int er = nb * R::BB;
  // L2 prefetch of output row d's bytes: shared down row and every used expert's row
  auto prefetch = [&](int d) {
    if (d >= a.D) return;
    const int e = shfl(rc.used, lane);
    if (lane < rc.nu) {
      bool far;
      const uint8_t *p = expert_at(a, e, far);
      if (!far) bulk_prefetch_l2(p + 2 * a.gate_bytes + (int64_t)d * er, (uint32_t)er);
    }
    if (lane == 31 && a.Fs > 0) bulk_prefetch_l2(a.sd + (int64_t)d * a.Fs, (uint32_t)a.Fs * 2u);
  };
  prefetch(gw);
  prefetch(gw + nwork);
  for (int d = gw; d < a.D; d += nwork) {
    prefetch(d + 2 * nwork);
    // shared down row (bf16) . hs
    float ys[4] = {0.f, 0.f, 0.f, 0.f};
    if (a.Fs > 0) {
      const uint16_t *row = a.sd + (int64_t)d * a.Fs;
#pragma unroll 8
      for (int c = 8 * lane; c < a.Fs; c += 256) {
        float wf[8];
        bf16x8(__ldcs(reinterpret_cast<const uint4 *>(row + c)), wf);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (t >= a.T) break;
          const float4 h0 = *reinterpret_cast<const float4 *>(hs + t * a.Fs + c);
          const float4 h1 = *reinterpret_cast<const float4 *>(hs + t * a.Fs + c + 4);
          ys[t] = fmaf(wf[0], h0.x, ys[t]); ys[t] = fmaf(wf[1], h0.y, ys[t]);
          ys[t] = fmaf(wf[2], h0.z, ys[t]); ys[t] = fmaf(wf[3], h0.w, ys[t]);
          ys[t] = fmaf(wf[4], h1.x, ys[t]); ys[t] = fmaf(wf[5], h1.y, ys[t]);
          ys[t] = fmaf(wf[6], h1.z, ys[t]); ys[t] = fmaf(wf[7], h1.w, ys[t]);
        }
      }
    }
    // every used expert's down row . its pairs' h (T <= 4 pairs per expert)
    float yreg = 0.f;  // lane p: y of pair p at this row
    constexpr int BATCH = 6;
    for (int u0 = 0; u0 < rc.nu; u0 += BATCH) {
      typename R::Row rp[BATCH];
#pragma unroll
      for (int v = 0; v < BATCH; ++v) {
        const int e = shfl(rc.used, min(u0 + v, 31));
        if (u0 + v < rc.nu) {
          bool far;
          R::load_g(expert_at(a, e, far) + 2 * a.gate_bytes + (int64_t)d * er, rp[v]);
        }
      }
      for (int j = 0; j < a.T; ++j) {  // j-th pair of every expert of the batch
        float y[BATCH];
#pragma unroll
        for (int v = 0; v < BATCH; ++v) {
          const int base = shfl(rc.base, min(u0 + v, 31)), n = shfl(rc.cnt, min(u0 + v, 31));
          y[v] = 0.f;
          if (u0 + v < rc.nu && j < n) {
            const uint32_t *pl = hpl + (base + j) * hw;
            y[v] = R::dot(rp[v], pl, reinterpret_cast<const float *>(pl + R::NPL * nsb), nsb);
          }
        }
        warp_sum_n<BATCH>(y);
#pragma unroll
        for (int v = 0; v < BATCH; ++v) {
          const int base = shfl(rc.base, min(u0 + v, 31)), n = shfl(rc.cnt, min(u0 + v, 31));
          const int pr = shfl(rc.perm, min(base + j, 31));
          if (u0 + v < rc.nu && j < n && lane == pr) yreg = y[v];
        }
      }
    }
    {
      float yst[4] = {ys[0], ys[1], ys[2], ys[3]};
      warp_sum_n<4>(yst);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (t >= a.T) break;
        float acc = yst[t];  // y_shared (0 without a shared expert)
        for (int j = 0; j < a.k; ++j) {
          const int p = t * a.k + j;
          acc = fmaf(shflf(rc.w, p), shflf(yreg, p), acc);
        }
        if (lane == 0) {
          float *o = a.out + (int64_t)t * a.D + d;
          *o = a.accumulate ? *o + acc : acc;
        }
      }
    }
  }
}

// ============================================================== one token ==
// The layer for one token in one cooperative kernel that streams every weight
// byte it needs through a ring of shared-memory stages filled by the
// bulk-copy engine, so that each SM keeps S_NS * S_STAGE bytes in flight.
//
//   phase A  tiles of gate/up rows: the shared expert two rows f, f+1 of
//            gate and up at a time, then every selected expert S_GU rows of
//            gate and up at a time -> h (routed, slot order) and hs (shared);
//   grid barrier (all of h is needed by every output row);
//   phase B  tiles of rb output rows d: the shared down rows and the rows of
//            every selected expert's down matrix -> out[d] = y_shared +
//            sum_j w_j y_j (pair order j).
//
// Warps 0..S_CONS-1 consume the stages (the same tile sequence on every
// warp, so their named barriers always match), warp S_CONS (one lane) issues
// the bulk copies and runs ahead across the grid barrier, warp S_CONS+1 waits
// for the router logits and selects the experts.  Every wait is bounded
// (S_LIMIT_NS); an expired wait sets ST_TIMEOUT and the kernel winds down
// without writing the output.
constexpr int S_CONS = 12;                       // consumer warps
constexpr int S_THREADS = (S_CONS + 2) * 32;     // + producer warp + router warp
// Registers per thread: four streaming warps of an SM sub-partition take
// 4 * 32 * 112 = 14,336 of its 16,384 registers, which leaves room for two
// warps of a router CTA at 32 registers (route_kernel's bounds), so the
// streaming grid's dependent launch starts while the router grid still runs.
// (Q2_K rows; the Q4_K kernels keep 128, which their rows need.)
constexpr int S_REGS = 112;
constexpr uint32_t S_STAGE = 32768;              // bytes per ring stage
constexpr int S_NS = 3;                          // ring stages
constexpr int S_GU = S_CONS;                     // routed gate/up rows per tile (one per warp)
constexpr int S_MAXP = 64;                       // slots x rows of a phase-B tile
constexpr int S_MAXK = 8;                        // top-k at most
constexpr int S_MAXT = 16;                       // shared or phase-B tiles of one block
constexpr uint64_t S_LIMIT_NS = WAIT_LIMIT_NS;    // bound of every wait

struct StreamShared {
  uint64_t full[S_NS], empty[S_NS];
  int rt_used[32];     // slot u -> expert (ascending expert id)
  int rt_pos[32];      // pair j -> its slot
  float rt_w[32];      // pair j -> routing weight
  int rt_nu;           // slots in use
  int ready;           // the route above is published
  int abort_;          // a wait expired
  int go;              // consumers continue past the grid barrier
  int tile[S_NS];                  // phase-A tile in each stage: shared i >= 0, routed -1 - (slot << 16 | row group)
  float reda[S_MAXT][S_CONS][4];   // per shared tile: partial gate/up sums of each warp
  float redb[S_MAXT][S_CONS][4];   // per phase-B tile: partial shared-down sums of each warp
  float yrb[S_MAXT][S_MAXP];       // per phase-B tile: routed down results [slot * rb + row]
};

__device__ __forceinline__ int vload(const int *p) { return *(volatile const int *)p; }

// Bounded wait for the phase of `bar` with parity `par`; false if it expired
// (flags ST_TIMEOUT) or another role of the block gave up.
__device__ bool s_wait(uint64_t *bar, uint32_t par, StreamShared &S, unsigned *status) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, par, 20000u)) {  // sleeps until the phase completes (20 us at most)
    if (vload(&S.abort_)) return false;
    if (globaltimer_ns() - t0 > wait_limit()) {
      flag(status, ST_TIMEOUT);
      *(volatile int *)&S.abort_ = 1;
      return false;
    }
  }
  return true;
}

// One row of an expert that has no cache slot, copied by the calling warp
// from host memory into its place in the stage (coalesced 16-byte loads; the
// producer copied nothing into that place), so that the dot reads it like a
// copied row.  One chunk per lane at a time keeps the registers of the
// streaming path free.  The proxy fence orders these stores before the bulk
// copies that later refill the stage.
__device__ __forceinline__ void warp_copy_row(const uint8_t *g, uint8_t *s, int bytes) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int o = 16 * lane; o < bytes; o += 512)
    *reinterpret_cast<uint4 *>(s + o) = __ldcs(reinterpret_cast<const uint4 *>(g + o));
  fence_proxy_async();
  __syncwarp();
}

// Bounded wait (one thread) for the route to be published.
__device__ bool s_wait_ready(StreamShared &S, unsigned *status) {
  const uint64_t t0 = globaltimer_ns();
  while (!vload(&S.ready)) {
    if (vload(&S.abort_)) return false;
    if (globaltimer_ns() - t0 > wait_limit()) {
      flag(status, ST_TIMEOUT);
      *(volatile int *)&S.abort_ = 1;
      return false;
    }
    __nanosleep(64);
  }
  __threadfence_block();
  return true;
}

__host__ __device__ constexpr size_t s_align(size_t v) { return (v + 127) & ~(size_t)127; }

__device__ __forceinline__ int tiles_of(int n, int bid, int G) { return bid < n ? (n - bid + G - 1) / G : 0; }

// Row format of the streaming kernel for an expert format: block bytes,
// weights per sub-block, planes per sub-block and the ring stage size (a
// routed gate/up tile, S_GU rows of gate and of up, fills one stage).
struct StreamFmt {
  int bb, sub, npl;
  uint32_t stage;
};
constexpr uint32_t S_STAGE_Q4 = 2 * S_GU * 16 * Q4B;  // 55,296 B: 12 gate + 12 up Q4_K rows of 4096
__host__ __device__ constexpr StreamFmt stream_fmt(int fmt) {
  return fmt == DS_Q4_K ? StreamFmt{Q4B, 32, 17, S_STAGE_Q4} : StreamFmt{QB, 16, 9, S_STAGE};
}

// Dynamic shared memory of the streaming kernel: stages, the small state,
// then one region used as x (phase A) and as h, hs (phase B).
size_t stream_smem(int fmt, int D, int F, int Fs, int nslots) {
  const StreamFmt f = stream_fmt(fmt);
  const size_t xa = 4 * (size_t)D + 4 * (f.npl * (size_t)(D / f.sub) + D / QK);
  const size_t hb = 4 * (size_t)nslots * (f.npl * (F / f.sub) + F / QK) + 4 * (size_t)Fs;
  return (size_t)S_NS * f.stage + s_align(sizeof(StreamShared)) + std::max(xa, hb);
}

// Rows per phase-B tile: the largest of 4, 2, 1 whose shared and routed down
// rows fit one stage.
int stream_rows_b(int fmt, int D, int F, int Fs, int nslots) {
  const StreamFmt f = stream_fmt(fmt);
  const int64_t rowb_f = (int64_t)(F / QK) * f.bb;
  for (int rb = 4; rb >= 1; rb >>= 1)
    if (D % rb == 0 && (int64_t)rb * nslots <= S_MAXP &&
        (int64_t)rb * (2 * (int64_t)Fs + nslots * rowb_f) <= f.stage)
      return rb;
  return 0;
}

// RD, RF: the row formats (Q2Rows / Q4Rows) of n_embd-long and n_ff-long
// rows; STG: the ring stage size.
template <class RD, class RF, uint32_t STG>
__global__ void __maxnreg__(RD::BB == QB ? S_REGS : 128) stream_kernel(const Args a, int rb) {
  // the next layer's router grid may launch now: it waits for this grid's
  // completion before it reads x or writes the workspace
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *stages = smem;
  StreamShared &S = *reinterpret_cast<StreamShared *>(smem + (size_t)S_NS * STG);
  uint8_t *reg = smem + (size_t)S_NS * STG + s_align(sizeof(StreamShared));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  const int D = a.D, F = a.F, Fs = a.Fs;
  const int nb_d = D / QK, nsb_d = D / RD::SUB, nb_f = F / QK, nsb_f = F / RF::SUB;
  const int rowb_d = nb_d * RD::BB, rowb_f = nb_f * RF::BB;
  const int nsa = Fs / 2;                       // shared gate/up tiles
  const int ngrp = (F + S_GU - 1) / S_GU;       // routed gate/up tiles per slot
  const int nslots = a.n_slots;
  const int nB = D / rb;
  const int lrb = 31 - __clz(rb);  // rb is 1, 2 or 4: pair p is (slot p >> lrb, row p & (rb - 1))
  // this block's phase-A tiles; routed tiles are dealt from the last block
  // down, so the blocks with one shared tile fewer get one routed tile more
  const int rbid = G - 1 - bid;
  const int ns_b = tiles_of(nsa, bid, G), nr_b = tiles_of(nslots * ngrp, rbid, G);
  const int nb_b = tiles_of(nB, bid, G);                                          // and phase-B tiles
  const int hw = RF::NPL * nsb_f + nb_f;
  constexpr int NT = S_CONS * 32;               // consumer threads
  float *xraw = reinterpret_cast<float *>(reg);                    // phase A
  uint32_t *xpl = reinterpret_cast<uint32_t *>(reg + 4 * (size_t)D);
  uint32_t *hpl = reinterpret_cast<uint32_t *>(reg);               // phase B
  float *hsm = reinterpret_cast<float *>(reg + 4 * (size_t)nslots * hw);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S_NS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], S_CONS);
    }
    S.ready = 0;
    S.abort_ = 0;
    S.go = 0;
    S.rt_nu = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- router --
  if (warp == S_CONS + 1) {
    pdl_wait();  // router logits complete and visible
    const RouteCache r = select_route_warp<S_MAXK>(a, bid == 0);  // one token: k pairs
    S.rt_used[lane] = r.used;
    S.rt_pos[lane] = r.pos;
    S.rt_w[lane] = r.w;
    if (lane == 0) S.rt_nu = r.nu;
    __threadfence_block();
    __syncwarp();
    if (lane == 0 && !hold_route()) *(volatile int *)&S.ready = 1;
    return;
  }

  // -------------------------------------------------------------- producer --
  if (warp == S_CONS) {
    if (lane != 0) return;
    int kq = 0;
    bool ok = true;
    // a free stage for the next tile (its previous tile consumed)
    auto acquire = [&]() -> uint8_t * {
      const int st = kq % S_NS;
      if (kq >= S_NS && !s_wait(&S.empty[st], ((kq / S_NS) & 1) ^ 1, S, a.status)) return nullptr;
      return stages + (size_t)st * STG;
    };
    // phase A: shared tiles while the route is pending, then shared and
    // routed tiles interleaved in proportion; the order is published per
    // stage in S.tile for the consumers
    bool have_route = false;
    for (int js = 0, jr = 0; ok && (js < ns_b || jr < nr_b);) {
      uint8_t *dst = acquire();
      if (!dst) { ok = false; break; }
      const int st = kq % S_NS;
      uint64_t *full = &S.full[st];
      if (!have_route) have_route = vload(&S.ready) != 0;
      const bool shared = js < ns_b && (!have_route || jr >= nr_b || (int64_t)js * nr_b <= (int64_t)jr * ns_b);
      if (shared) {
        const int i = bid + G * js++;
        S.tile[st] = i;
        const uint32_t bytes = 4u * (uint32_t)D;  // rows f, f+1 in bf16
        mbar_arrive_expect_tx(full, 2 * bytes);
        bulk_g2s(dst, a.sg + (size_t)(2 * i) * D, bytes, full);
        bulk_g2s(dst + bytes, a.su + (size_t)(2 * i) * D, bytes, full);
      } else {
        if (!have_route && !(have_route = s_wait_ready(S, a.status))) { ok = false; break; }
        const int r = rbid + G * jr++, u = r / ngrp, g = r % ngrp;
        S.tile[st] = -1 - ((u << 16) | g);  // the consumers take u and g without a division
        const int rows = min(S_GU, F - g * S_GU);
        bool far = false;
        const uint8_t *gr = u < S.rt_nu ? expert_at(a, S.rt_used[u], far) + (int64_t)g * S_GU * rowb_d : nullptr;
        if (u < S.rt_nu && !far) {
          const uint32_t bytes = (uint32_t)(rows * rowb_d);
          mbar_arrive_expect_tx(full, 2 * bytes);
          bulk_g2s(dst, gr, bytes, full);
          bulk_g2s(dst + S_GU * rowb_d, gr + a.gate_bytes, bytes, full);
        } else {
          mbar_arrive(full);  // nothing to copy (an expert in host memory: the consumers load its rows)
        }
      }
      ++kq;
    }
    // phase B needs no h: its copies run ahead across the grid barrier
    for (int m = 0; ok && m < nb_b; ++m) {
      if (!have_route && !(have_route = s_wait_ready(S, a.status))) break;
      uint8_t *dst = acquire();
      if (!dst) break;
      uint64_t *full = &S.full[kq % S_NS];
      const int d0 = (bid + G * m) * rb, nu = S.rt_nu;
      const uint32_t sb = (uint32_t)(rb * 2 * Fs), ub = (uint32_t)(rb * rowb_f);
      uint32_t near_bytes = 0;
      for (int u = 0; u < nu; ++u) {
        bool far;
        (void)expert_at(a, S.rt_used[u], far);
        if (!far) near_bytes += ub;
      }
      mbar_arrive_expect_tx(full, sb + near_bytes);
      if (Fs > 0) bulk_g2s(dst, a.sd + (size_t)d0 * Fs, sb, full);
      for (int u = 0; u < nu; ++u) {
        bool far;
        const uint8_t *p = expert_at(a, S.rt_used[u], far);
        if (!far) bulk_g2s(dst + sb + (size_t)u * ub, p + 2 * a.gate_bytes + (int64_t)d0 * rowb_f, ub, full);
      }
      ++kq;
    }
    // keep the block resident until every copy issued has landed
    for (int q = kq > S_NS ? kq - S_NS : 0; q < kq; ++q) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&S.full[q % S_NS], (q / S_NS) & 1))
        if (globaltimer_ns() - t0 > S_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
    }
    return;
  }

  // ------------------------------------------------------------- consumers --
  // x as fp32 (shared-expert rows) and as fixed-point planes (Q2_K rows),
  // one half-warp per 256-element block, all loads in one round (from the
  // router grid's device copy when x is in host memory)
  const void *xin = a.x;
  if (a.x_stage) {
    pdl_wait();
    xin = a.x_stage;
  }
  for (int u = warp; u < (nb_d + 1) / 2; u += S_CONS) {
    const int blk = min(2 * u + (lane >> 4), nb_d - 1);
    const int64_t e0 = (int64_t)QK * blk + 16 * (lane & 15);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = a.x_f32 ? __ldg((const float *)xin + e0 + j) : bf16_to_f32(__ldg((const uint16_t *)xin + e0 + j));
#pragma unroll
    for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4 *>(xraw + e0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    RD::digitize(v, blk, xpl, reinterpret_cast<float *>(xpl + RD::NPL * nsb_d), nsb_d);
  }
  named_bar(1, NT);
  int nu = 0;
  {
    typename RD::XR xr;
    RD::load_x(xpl, reinterpret_cast<const float *>(xpl + RD::NPL * nsb_d), nsb_d, xr);
    bool have_route = false;
    int js = 0;
    for (int kq = 0; kq < ns_b + nr_b; ++kq) {
      const int st = kq % S_NS;
      const bool got = s_wait(&S.full[st], (kq / S_NS) & 1, S, a.status);
      const uint8_t *src = stages + (size_t)st * STG;
      const int td = got ? S.tile[st] : 0;
      if (td >= 0) {
        // rows in the stage: gate f, gate f+1, up f, up f+1; every consumer
        // thread takes eight-element chunks of all four rows (x read once)
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (got) {
          for (int c = 8 * threadIdx.x; c < D; c += 8 * NT) {
            const float4 x0 = *reinterpret_cast<const float4 *>(xraw + c);
            const float4 x1 = *reinterpret_cast<const float4 *>(xraw + c + 4);
#pragma unroll
            for (int row = 0; row < 4; ++row) {
              float wf[8];
              bf16x8(*reinterpret_cast<const uint4 *>(src + (size_t)row * 2 * D + 2 * (size_t)c), wf);
              float t = acc[row];
              t = fmaf(wf[0], x0.x, t); t = fmaf(wf[1], x0.y, t); t = fmaf(wf[2], x0.z, t); t = fmaf(wf[3], x0.w, t);
              t = fmaf(wf[4], x1.x, t); t = fmaf(wf[5], x1.y, t); t = fmaf(wf[6], x1.z, t); t = fmaf(wf[7], x1.w, t);
              acc[row] = t;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[st]);
        const float tot = warp_sum_spread<4>(acc);  // lane 8 row: total of row
        if ((lane & 7) == 0 && js < S_MAXT) S.reda[js][warp][lane >> 3] = tot;
        ++js;
        continue;
      }
      if (!have_route) {
        int rdy = 1;
        if (lane == 0) rdy = s_wait_ready(S, a.status) ? 1 : 0;
        rdy = __shfl_sync(0xffffffffu, rdy, 0);
        __threadfence_block();
        nu = rdy ? S.rt_nu : 0;
        have_route = true;
      }
      const int ug = -1 - td, u = ug >> 16, g = ug & 0xFFFF;
      const int f = g * S_GU + warp;
      if (got && u < nu && f < F) {
        typename RD::Row gp, up;
        bool far;
        const uint8_t *hrow = expert_at(a, S.rt_used[u], far) + (int64_t)f * rowb_d;
        if (far) {  // the expert's rows, from host memory into their place in the stage
          warp_copy_row(hrow, const_cast<uint8_t *>(src) + (size_t)warp * rowb_d, rowb_d);
          warp_copy_row(hrow + a.gate_bytes, const_cast<uint8_t *>(src) + (size_t)(S_GU + warp) * rowb_d, rowb_d);
        }
        RD::load_s(src + (size_t)warp * rowb_d, gp);
        RD::load_s(src + (size_t)(S_GU + warp) * rowb_d, up);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[st]);
        const float gu[2] = {RD::dot_reg(gp, xr), RD::dot_reg(up, xr)};
        const float tot = warp_sum_spread<2>(gu);  // lane 0: gate, lane 16: up
        const float upv = __shfl_sync(0xffffffffu, tot, 16);
        if (lane == 0) a.h[(int64_t)u * F + f] = silu(tot) * upv;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[st]);
      }
    }
  }
  // hs of this block's shared tiles: gate and up summed over the warps in
  // a fixed order
  named_bar(1, NT);
  for (int t = threadIdx.x; t < 2 * min(ns_b, S_MAXT); t += NT) {
    const int m = t >> 1, h = t & 1;
    float g = 0.f, u = 0.f;
    for (int w = 0; w < S_CONS; ++w) {
      g += S.reda[m][w][h];
      u += S.reda[m][w][2 + h];
    }
    a.hs[2 * (bid + G * m) + h] = silu(g) * u;
  }

  // grid barrier: every block's h and hs are written
  named_bar(1, NT);
  if (threadIdx.x == 0) {
    bool fine = !vload(&S.abort_) && s_wait_ready(S, a.status);
    if (fine) {
      pdl_wait();  // the router grid (which reset the barrier word) has completed
      // the release add publishes every h and hs store of the block: they
      // precede this thread's add through the named barrier above
      atom_add_release(a.ctrl + C_BAR, 1u);
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(a.ctrl + C_BAR) < (unsigned)G) {
        if (globaltimer_ns() - t0 > wait_limit()) {
          flag(a.status, ST_TIMEOUT);
          fine = false;
          break;
        }
      }
    }
    if (!fine) *(volatile int *)&S.abort_ = 1;
    S.go = fine ? 1 : 0;  // the one decision every consumer warp follows
  }
  named_bar(1, NT);
  if (!vload(&S.go)) return;
  nu = S.rt_nu;

  // h of every slot in fixed point, and hs: one half-warp per 256-element
  // block, two blocks per half-warp and pass, with the hs loads and every h
  // load of the pass issued before the first use
  {
    constexpr int HSR = 8;  // hs values per thread kept in flight
    float hv[HSR];
#pragma unroll
    for (int j = 0; j < HSR; ++j) {
      const int i = threadIdx.x + j * NT;
      hv[j] = i < Fs ? __ldcg(a.hs + i) : 0.f;
    }
    const int nblk = nu * nb_f, nun = (nblk + 1) / 2;
    for (int un = warp; un < nun; un += 2 * S_CONS) {
      float v[2][16];
      int q[2], blk[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int bi = min(2 * min(un + h * S_CONS, nun - 1) + (lane >> 4), nblk - 1);
        q[h] = bi / nb_f;
        blk[h] = bi % nb_f;
        const float4 *hsrc = reinterpret_cast<const float4 *>(a.h + (int64_t)q[h] * F + QK * blk[h] + 16 * (lane & 15));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 f4 = __ldcg(hsrc + j);
          v[h][4 * j] = f4.x; v[h][4 * j + 1] = f4.y; v[h][4 * j + 2] = f4.z; v[h][4 * j + 3] = f4.w;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
        RF::digitize(v[h], blk[h], hpl + q[h] * hw, reinterpret_cast<float *>(hpl + q[h] * hw + RF::NPL * nsb_f), nsb_f);
    }
#pragma unroll
    for (int j = 0; j < HSR; ++j) {
      const int i = threadIdx.x + j * NT;
      if (i < Fs) hsm[i] = hv[j];
    }
    for (int i = threadIdx.x + HSR * NT; i < Fs; i += NT) hsm[i] = __ldcg(a.hs + i);
  }
  named_bar(1, NT);

  // phase B: every consumer thread takes eight-element chunks of all rb
  // shared rows (hs read once); warp w takes the routed (slot, row) pairs
  // 2w and 2w + 1 when there are at most two per warp — with rb even both
  // rows belong to one slot, whose h planes the warp then loads into
  // registers once — else it loops over its pairs one at a time
  const int np = nu * rb;
  const bool two = np <= 2 * S_CONS;
  int kq = ns_b + nr_b;
  for (int m = 0; m < nb_b; ++m, ++kq) {
    const int st = kq % S_NS;
    const bool got = s_wait(&S.full[st], (kq / S_NS) & 1, S, a.status);
    const uint8_t *src = stages + (size_t)st * STG;
    float ys[4] = {0.f, 0.f, 0.f, 0.f};
    if (got) {
      for (int c = 8 * threadIdx.x; c < Fs; c += 8 * NT) {
        const float4 h0 = *reinterpret_cast<const float4 *>(hsm + c);
        const float4 h1 = *reinterpret_cast<const float4 *>(hsm + c + 4);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (r >= rb) break;
          float wf[8];
          bf16x8(*reinterpret_cast<const uint4 *>(src + (size_t)r * 2 * Fs + 2 * (size_t)c), wf);
          float t = ys[r];
          t = fmaf(wf[0], h0.x, t); t = fmaf(wf[1], h0.y, t); t = fmaf(wf[2], h0.z, t); t = fmaf(wf[3], h0.w, t);
          t = fmaf(wf[4], h1.x, t); t = fmaf(wf[5], h1.y, t); t = fmaf(wf[6], h1.z, t); t = fmaf(wf[7], h1.w, t);
          ys[r] = t;
        }
      }
    }
    const uint8_t *routed = src + (size_t)rb * 2 * Fs;
    // pair p = (slot p / rb, row p % rb) of this tile: from the stage, or from
    // host memory for an expert that has no cache slot
    auto load_down_row = [&](int p, typename RF::Row &row) {
      bool far;
      const uint8_t *hp = expert_at(a, S.rt_used[p >> lrb], far);
      if (far)
        warp_copy_row(hp + 2 * a.gate_bytes + (int64_t)((bid + G * m) * rb + (p & (rb - 1))) * rowb_f,
                      const_cast<uint8_t *>(routed) + (size_t)p * rowb_f, rowb_f);
      RF::load_s(routed + (size_t)p * rowb_f, row);
    };
    float y[2] = {0.f, 0.f};
    if (two) {
      typename RF::Row rp[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = 2 * warp + h;
        if (got && p < np) load_down_row(p, rp[h]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      if (got && 2 * warp < np) {
        if ((rb & 1) == 0) {  // one slot: its planes in registers, two dots
          const uint32_t *pl = hpl + ((2 * warp) >> lrb) * hw;
          typename RF::XR hr;
          RF::load_x(pl, reinterpret_cast<const float *>(pl + RF::NPL * nsb_f), nsb_f, hr);
          y[0] = RF::dot_reg(rp[0], hr);
          y[1] = RF::dot_reg(rp[1], hr);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int p = 2 * warp + h;
            if (p < np) {
              const uint32_t *pl = hpl + (p >> lrb) * hw;
              y[h] = RF::dot(rp[h], pl, reinterpret_cast<const float *>(pl + RF::NPL * nsb_f), nsb_f);
            }
          }
        }
      }
      const float v8[8] = {ys[0], ys[1], ys[2], ys[3], y[0], y[1], 0.f, 0.f};
      const float tot = warp_sum_spread<8>(v8);  // lane 4 i: total of v8[i]
      const int vi = lane >> 2;
      if ((lane & 3) == 0 && m < S_MAXT) {
        if (vi < 4) S.redb[m][warp][vi] = tot;
        else if (vi < 6 && 2 * warp + (vi - 4) < np) S.yrb[m][2 * warp + (vi - 4)] = tot;
      }
    } else {
      // one pair at a time, the stage released after the last
      warp_sum_n<4>(ys);
      if (lane == 0 && m < S_MAXT) {
#pragma unroll
        for (int r = 0; r < 4; ++r) S.redb[m][warp][r] = ys[r];
      }
      for (int p = warp; p < np; p += S_CONS) {
        float yy = 0.f;
        if (got) {
          typename RF::Row rp;
          load_down_row(p, rp);
          const uint32_t *pl = hpl + (p >> lrb) * hw;
          yy = RF::dot(rp, pl, reinterpret_cast<const float *>(pl + RF::NPL * nsb_f), nsb_f);
        }
        yy = warp_sum(yy);
        if (lane == 0 && m < S_MAXT) S.yrb[m][p] = yy;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
    }
  }
  // the combine of this block's output rows: y_shared (summed over the warps
  // in a fixed order) + sum_j w_j y_j in pair order j
  named_bar(1, NT);
  if (vload(&S.abort_)) return;
  for (int t = threadIdx.x; t < min(nb_b, S_MAXT) * rb; t += NT) {
    const int m = t / rb, r = t % rb;
    float acc = 0.f;
    for (int w = 0; w < S_CONS; ++w) acc += S.redb[m][w][r];
    for (int j = 0; j < a.k; ++j) acc = fmaf(S.rt_w[j], S.yrb[m][S.rt_pos[j] * rb + r], acc);
    float *o = a.out + (int64_t)(bid + G * m) * rb + r;
    *o = a.accumulate ? *o + acc : acc;
  }
}

size_t k2_smem(int fmt, int T, int D) {
  const StreamFmt f = stream_fmt(fmt);
  return 4 * (size_t)T * (f.npl * (D / f.sub) + D / QK);
}
size_t k3_smem(int fmt, int T, int k, int F, int Fs) {
  const StreamFmt f = stream_fmt(fmt);
  return 4 * ((size_t)T * k * (f.npl * (F / f.sub) + F / QK) + (size_t)T * Fs);
}

template <typename K>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Args &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class RD, class RF>
cudaError_t launch_all(const Args &a, const Shape &sh, cudaStream_t s) {
  static OncePerDevice once;
  const int sms = device_sms();
  if (!sms) return cudaErrorNoDevice;
  cudaError_t e = once_per_device(once, []() {  // dynamic caps leave room for the kernels' static shared memory
    cudaError_t r = cudaFuncSetAttribute(gateup_kernel<RD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(SMEM_LIMIT - 4096));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(down_kernel<RF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(SMEM_LIMIT - 4096));
    return r;
  });
  if (e != cudaSuccess) return e;
  const dim3 g1((sh.E + 1) / 2);
  if (sh.x_dtype == DS_BF16 && sh.router_dtype == DS_BF16) e = launch_pdl(route_kernel<uint16_t, uint16_t>, g1, dim3(256), 0, s, a);
  else if (sh.x_dtype == DS_F32 && sh.router_dtype == DS_F32) e = launch_pdl(route_kernel<float, float>, g1, dim3(256), 0, s, a);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(gateup_kernel<RD>, dim3(sms), dim3(NW2 * 32), k2_smem(sh.fmt, a.T, a.D), s, a)) != cudaSuccess)
    return e;
  return launch_pdl(down_kernel<RF>, dim3(sms), dim3(NW3 * 32), k3_smem(sh.fmt, a.T, a.k, a.F, a.Fs), s, a);
}

// One token: router logits, then the streaming kernel (cooperative, so the
// grid barrier is safe; PDL lets its prologue overlap the router grid).
template <class RD, class RF, uint32_t STG>
cudaError_t launch_stream(const Args &a, const Shape &sh, int rb, cudaStream_t s) {
  static OncePerDevice once;
  const int sms = device_sms();
  if (!sms) return cudaErrorNoDevice;
  const size_t smem = stream_smem(sh.fmt, a.D, a.F, a.Fs, a.n_slots);
  cudaError_t e0 = once_per_device(once, []() {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<RD, RF, STG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    // the router grid runs with the streaming kernel's shared-memory split,
    // so that the SMs need no reconfiguration between the two
    for (const void *f : {(const void *)route_kernel<uint16_t, uint16_t>, (const void *)route_kernel<float, float>,
                          (const void *)stream_kernel<RD, RF, STG>})
      if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
        return e;
    return cudaSuccess;
  });
  if (e0 != cudaSuccess) return e0;
  // the grid barrier needs every block resident: one block per SM at this
  // call's shared-memory size (checked per device and size)
  {
    static std::mutex mu;
    static int dev_seen[64] = {};
    static size_t smem_seen[64] = {};
    int dev = 0;
    if ((e0 = cudaGetDevice(&dev)) != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!dev_seen[dev] || smem_seen[dev] != smem) {
      int per_sm = 0;
      e0 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel<RD, RF, STG>, S_THREADS, smem);
      if (e0 != cudaSuccess) return e0;
      if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
      dev_seen[dev] = 1;
      smem_seen[dev] = smem;
    }
  }
  const dim3 g1((sh.E + 1) / 2);
  cudaError_t e;
  if (sh.x_dtype == DS_BF16 && sh.router_dtype == DS_BF16) e = launch_pdl(route_kernel<uint16_t, uint16_t>, g1, dim3(256), 0, s, a);
  else if (sh.x_dtype == DS_F32 && sh.router_dtype == DS_F32) e = launch_pdl(route_kernel<float, float>, g1, dim3(256), 0, s, a);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(S_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, stream_kernel<RD, RF, STG>, a, rb);
  if (e != cudaSuccess) {  // without the overlap: plain stream order
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, stream_kernel<RD, RF, STG>, a, rb);
  }
  return e;
}

}  // namespace

// (n_embd / 256, n_ff / 256) with instantiated kernels
static bool fast_shape_ok(int nb_d, int nb_f) {
  return (nb_d == 16 && nb_f == 8) || (nb_d == 4 && nb_f == 4);
}

// Shape conditions shared by the three-kernel chain and the streaming kernel.
static bool fused_shape_ok(const Shape &sh, int64_t T) {
  if (T < 1 || T > 4 || (int64_t)T * sh.k > PMAXD) return false;
  if (sh.D % QK || sh.F % QK || !fast_shape_ok(sh.D / QK, sh.F / QK)) return false;
  if (sh.x_dtype != sh.router_dtype || sh.E > 1024) return false;
  // the shared partial sums [2][4][T][Fs] live in the routed-output region [T*k][D]
  if ((int64_t)8 * sh.Fs > (int64_t)sh.k * sh.D) return false;
  return true;
}

bool fused_decode_supported(const Shape &sh, int64_t T) {
  if ((sh.fmt != DS_Q2_K && sh.fmt != DS_Q4_K) || !fused_shape_ok(sh, T)) return false;
  return k2_smem(sh.fmt, (int)T, sh.D) <= SMEM_LIMIT - 4096 &&
         k3_smem(sh.fmt, (int)T, sh.k, sh.F, sh.Fs) <= SMEM_LIMIT - 4096;
}

bool stream_decode_supported(const Shape &sh, int64_t T) {
  if (T != 1 || sh.k > S_MAXK || !fused_shape_ok(sh, T)) return false;
  const int nb_d = sh.D / QK, nb_f = sh.F / QK, nslots = std::min(sh.E, sh.k);
  const StreamFmt f = stream_fmt(sh.fmt);
  const int rb = stream_rows_b(sh.fmt, sh.D, sh.F, sh.Fs, nslots);
  const int sms = device_sms();
  return rb > 0 && sms > 0 && stream_smem(sh.fmt, sh.D, sh.F, sh.Fs, nslots) <= SMEM_LIMIT && nslots <= 32 &&
         8 * (int64_t)sh.D <= f.stage && 2 * S_GU * (int64_t)nb_d * f.bb <= f.stage && nb_f % 4 == 0 &&
         (sh.Fs / 2 + sms - 1) / sms <= S_MAXT && (sh.D / rb + sms - 1) / sms <= S_MAXT;
}

cudaError_t launch_decode_fused(const Shape &sh, const ds_moe_weights &W, const void *x,
                                const Work &wk, float *out, bool accumulate, cudaStream_t s, void *x_stage,
                                const Residency *res) {
  Args a{};
  a.D = sh.D; a.E = sh.E; a.F = sh.F; a.Fs = sh.Fs; a.k = sh.k; a.T = (int)wk.T;
  a.routed_scale = sh.routed_scale;
  a.logit_scale = sh.logit_scale;
  a.bias_select_only = sh.bias_select_only;
  a.router_w = W.router_w;
  a.router_f32 = sh.router_dtype == DS_F32;
  a.bias = W.router_bias;
  a.sg = W.shared_gate; a.su = W.shared_up; a.sd = W.shared_down;
  a.experts = W.experts;
  a.expert_bytes = sh.expert_bytes();
  a.gate_bytes = sh.gate_bytes();
  if (res) {
    a.slot = res->slot;
    a.cache = res->cache;
    a.host = res->host;
  }
  a.x = x;
  a.x_f32 = sh.x_dtype == DS_F32;
  a.x_stage = nullptr;
  if (x_stage) {  // only the one-token kernel reads the staged copy
    if (!stream_decode_supported(sh, wk.T)) return cudaErrorInvalidValue;
    a.x_stage = x_stage;
  }
  a.logits = wk.logits; a.ids = wk.ids; a.w = wk.w;
  a.counts = wk.counts; a.offsets = wk.offsets; a.perm = wk.perm; a.pos = wk.pos; a.used = wk.used;
  a.h = wk.h;
  a.hs = wk.hs;
  a.pgu = wk.y;
  a.ctrl = wk.ctrl;
  a.out = out;
  a.accumulate = accumulate ? 1 : 0;
  a.status = status_word();
  a.n_slots = (int)std::min<int64_t>(sh.E, wk.T * sh.k);
  const int nb_d = sh.D / QK, nb_f = sh.F / QK;
  if (stream_decode_supported(sh, wk.T)) {
    const int rb = stream_rows_b(sh.fmt, a.D, a.F, a.Fs, a.n_slots);
    if (sh.fmt == DS_Q4_K) {
      if (nb_d == 16 && nb_f == 8) return launch_stream<Q4Rows<4>, Q4Rows<2>, S_STAGE_Q4>(a, sh, rb, s);
      if (nb_d == 4 && nb_f == 4) return launch_stream<Q4Rows<1>, Q4Rows<1>, S_STAGE_Q4>(a, sh, rb, s);
      return cudaErrorInvalidValue;
    }
    if (nb_d == 16 && nb_f == 8) return launch_stream<Q2Rows<8>, Q2Rows<4>, S_STAGE>(a, sh, rb, s);
    if (nb_d == 4 && nb_f == 4) return launch_stream<Q2Rows<2>, Q2Rows<2>, S_STAGE>(a, sh, rb, s);
  }
  if (sh.fmt == DS_Q4_K) {
    if (nb_d == 16 && nb_f == 8) return launch_all<Q4Rows<4>, Q4Rows<2>>(a, sh, s);
    if (nb_d == 4 && nb_f == 4) return launch_all<Q4Rows<1>, Q4Rows<1>>(a, sh, s);
    return cudaErrorInvalidValue;
  }
  if (nb_d == 16 && nb_f == 8) return launch_all<Q2Rows<8>, Q2Rows<4>>(a, sh, s);
  if (nb_d == 4 && nb_f == 4) return launch_all<Q2Rows<2>, Q2Rows<2>>(a, sh, s);
  return cudaErrorInvalidValue;
}

}  // namespace dsm

#ifdef DS_MOE_TEST_HOOKS
// Test build only: sets the hooks above on the current device (flags bit 0:
// hold the route; limit_ns: the shortened bound, 0 = the normal one).
extern "C" int ds_moe_test_hooks(unsigned flags, unsigned long long limit_ns) {
  cudaError_t e = cudaMemcpyToSymbol(dsm::g_test_hook_flags, &flags, sizeof flags);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dsm::g_test_hook_limit_ns, &limit_ns, sizeof limit_ns);
  return e == cudaSuccess ? 0 : -3;
}
#endif
