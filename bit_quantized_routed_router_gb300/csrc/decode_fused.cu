// Decode path for one token (T = 1 at the 4096/256/6/2048 shape; any shape
// whose staging fits shared memory): the whole layer in one persistent kernel.
//
// What it computes is the layer of "Understanding Dwarf Star" 5.3.2/5.3.7
// (router -> top-k -> gate/up -> SiLU(gate)*up -> down -> weighted sum, plus
// the always-active shared expert of 5.3.4), with the routed weights read as
// Q2_K blocks (3.3.3) and dequantised on the fly (2.8.1-2.8.2).
//
// How (GB300-first):
//  * One CTA per SM (cooperative launch: every CTA resident) of NW worker
//    warps.  Each worker is autonomous: it owns a ring of NS shared-memory
//    stages and one mbarrier per stage, issues 1-D bulk copies (TMA engine)
//    for its next chunks from lane 0, and consumes them; no CTA-wide barrier
//    is taken in the steady state.
//  * Tasks, dealt round-robin over all workers in this order:
//      router rows -> shared gate/up rows -> routed gate/up row groups
//      -> output rows (all experts' down rows + shared down row + combine).
//    A task waits only for earlier tasks (the route; all gate/up results),
//    every worker runs its tasks in order and all workers are resident, so
//    every wait ends; each wait is also bounded (2 s) and reports a timeout
//    through the status word instead of hanging.
//  * Chunks of later tasks are fetched while earlier ones compute, and the
//    down rows are fetched as soon as the route is known, so HBM stays busy
//    across the phase boundaries.
//  * Q2_K dot products are exact integer sums: activations are converted once
//    per 16-element sub-block to 24-bit fixed point X = rint(v / step),
//    step = 2^(e-23) with max|v| < 2^e, split into three bytes, and
//    sum_j q_j X_j is formed with dp4a; then w.x = step*(d*sc*S - dmin*m*sum X).
//    The only rounding beyond fp32 is that fixed point (|err| <= 2^-23 of the
//    sub-block's largest element).
//  * The last task of each output row adds y_shared + sum_j w_j y_j in slot
//    order j: no atomics in the values, deterministic results.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dsm {
namespace {

constexpr int NW = 16;                    // worker warps per CTA
constexpr int NTHREADS = NW * 32;
constexpr int SB = 2816;                  // bytes per stage: two 1344-byte Q2_K rows
constexpr int TMAXF = 2;                  // tokens this path serves
constexpr int PMAXF = TMAXF * 16;         // token-expert pairs
constexpr int RG = 4;                     // routed gate/up rows per task
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr size_t SMEM_LIMIT = 227 * 1024;

enum { C_ROUTER = 0, C_READY = 1, C_GU = 2, C_ABORT = 3, C_NUSED = 4 };
enum { K_ROUTER = 0, K_SGU = 1, K_RGU = 2, K_DOWN = 3 };

// Activations in fixed point, per 256-element super-block b (the Q2_K block):
//   X_j = rint(v_j / step_b), step_b = 2^(e_b - 15) with max_b |v| < 2^e_b,
//   clamped to |X_j| <= 32767, split as X = hi*256 + lo (hi signed byte,
//   lo unsigned byte).
// Planes: for sub-block sb, word i of hi (lo) holds the byte of X_{16 sb + 4c + i}
// in byte c -- the byte order of (codes >> 2i) & 0x03030303 -- so that
// sum_j q_j X_j = 256 * sum_i dp4a(q_i, hi_i) + sum_i dp4a(q_i, lo_i).
// Nine planes (hi0..3, lo0..3, SX = sum_j X_j) of nsb words each, followed by
// nb steps.  Within a plane, sub-blocks are stored in the order lanes read
// them (see lane_map), so each lane's vector load is conflict-free.
//
// Lane mapping for a Q2_K row of nb = 2..32 blocks: LPB = 32/nb lanes per
// block, SPL = nb/2 sub-blocks per lane; lane l takes block l / LPB and its
// sub-blocks SPL*(l % LPB) + i, i < SPL.
template <int SPL>
struct LaneMap {
  static constexpr int LPB = 16 / SPL;
  static constexpr int Q = SPL < 4 ? SPL : 4;  // words per vector load
  // plane offset (in words) of (lane, i)
  __device__ static __forceinline__ int off(int lane, int i) {
    return (i / Q) * (32 * Q) + lane * Q + (i % Q);
  }
  __device__ static __forceinline__ int sb(int lane, int i) {
    return 16 * (lane / LPB) + SPL * (lane % LPB) + i;
  }
};

// Convert one super-block (256 values, sub-block s = lane & 15 of the calling
// half-warp holds v[16]) into the planes.  Called by all 32 lanes for two
// blocks at once (lanes 0-15: block b0, 16-31: block b1).
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
  const float inv = m > 0.f ? ldexpf(1.0f, 15 - e) : 0.f;  // exact power of two
  uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
  int sx = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    int X = __float2int_rn(v[j] * inv);
    X = max(-32767, min(32767, X));
    sx += X;
    const int i = j & 3, c = 8 * (j >> 2);
    hi[i] |= ((uint32_t)(X >> 8) & 0xFFu) << c;
    lo[i] |= ((uint32_t)X & 0xFFu) << c;
  }
  // which lane reads this sub-block, and as which of its sub-blocks
  const int sb = 16 * b + s;
  const int l_read = (sb / 16) * LaneMap<SPL>::LPB + (sb % 16) / SPL;
  const int o = LaneMap<SPL>::off(l_read, (sb % 16) % SPL);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    planes[i * nsb + o] = hi[i];
    planes[(4 + i) * nsb + o] = lo[i];
  }
  planes[8 * nsb + o] = (uint32_t)sx;
  if (s == 0) steps[b] = m > 0.f ? ldexpf(1.0f, e - 15) : 0.f;
}

template <int Q>
__device__ __forceinline__ void ld_words(const uint32_t *p, uint32_t w[Q]) {
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

// This lane's part of (Q2_K row in shared memory) . (activation planes):
// integer sums over the lane's sub-blocks, two conversions to float at the end.
template <int SPL>
__device__ __forceinline__ float q2k_dot(const uint8_t *row, const uint32_t *planes,
                                         const float *steps, int nsb) {
  using M = LaneMap<SPL>;
  constexpr int Q = M::Q;
  const int lane = threadIdx.x & 31;
  const int b = lane / M::LPB, s0 = SPL * (lane % M::LPB);
  const uint8_t *blk = row + b * QB;
  int accq = 0, accm = 0;
#pragma unroll
  for (int g = 0; g < SPL / Q; ++g) {
    uint32_t hi[4][Q], lo[4][Q], sx[Q];
    const int o = g * (32 * Q) + lane * Q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ld_words<Q>(planes + i * nsb + o, hi[i]);
      ld_words<Q>(planes + (4 + i) * nsb + o, lo[i]);
    }
    ld_words<Q>(planes + 8 * nsb + o, sx);
#pragma unroll
    for (int k = 0; k < Q; ++k) {
      const int s = s0 + g * Q + k;
      const uint32_t codes = *reinterpret_cast<const uint32_t *>(blk + 16 + 4 * s);
      const int scm = blk[s];
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
      const int S = sh * 256 + (int)sl;  // sum_j q_j X_j over the sub-block, exact
      accq += (scm & 15) * S;
      accm += (scm >> 4) * (int)sx[k];
    }
  }
  const uint32_t dd = *reinterpret_cast<const uint32_t *>(blk + 80);
  const float d = fp16_to_f32((uint16_t)(dd & 0xFFFF)), dmin = fp16_to_f32((uint16_t)(dd >> 16));
  return steps[b] * fmaf(d, (float)accq, -dmin * (float)accm);
}

__device__ __forceinline__ void bf16x8(uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Dense row piece (shared memory, n elements of bf16 or fp32) . activation
// piece (global bf16/fp32, or shared fp32); lane covers elements 8 lane + 256 i.
__device__ __forceinline__ float dense_dot(const uint8_t *row, bool row_f32, int n, const void *xv,
                                           int x_kind /*0 bf16 gmem, 1 f32 gmem, 2 f32 smem*/) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int c = 8 * lane; c < n; c += 256) {
    float wf[8], xf[8];
    if (row_f32) {
      const float4 *p = reinterpret_cast<const float4 *>(row) + c / 4;
      const float4 a = p[0], b = p[1];
      wf[0] = a.x; wf[1] = a.y; wf[2] = a.z; wf[3] = a.w;
      wf[4] = b.x; wf[5] = b.y; wf[6] = b.z; wf[7] = b.w;
    } else {
      bf16x8(*reinterpret_cast<const uint4 *>(row + 2 * c), wf);
    }
    if (x_kind == 0) {
      bf16x8(__ldg(reinterpret_cast<const uint4 *>((const uint16_t *)xv + c)), xf);
    } else {
      const float4 *p = reinterpret_cast<const float4 *>((const float *)xv + c);
      const float4 a = x_kind == 1 ? __ldg(p) : p[0], b = x_kind == 1 ? __ldg(p + 1) : p[1];
      xf[0] = a.x; xf[1] = a.y; xf[2] = a.z; xf[3] = a.w;
      xf[4] = b.x; xf[5] = b.y; xf[6] = b.z; xf[7] = b.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], xf[i], acc);
  }
  return acc;
}

// bf16 row piece (shared memory) . fp32 activation piece (shared memory);
// lane covers elements 4 lane + 128 i, so both reads are conflict-free.
__device__ __forceinline__ float dense_dot_s(const uint8_t *row, int n, const float *xs) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int c = 4 * lane; c < n; c += 128) {
    const uint2 wv = *reinterpret_cast<const uint2 *>(row + 2 * c);
    const float4 xv = *reinterpret_cast<const float4 *>(xs + c);
    acc = fmaf(__uint_as_float(wv.x << 16), xv.x, acc);
    acc = fmaf(__uint_as_float(wv.x & 0xFFFF0000u), xv.y, acc);
    acc = fmaf(__uint_as_float(wv.y << 16), xv.z, acc);
    acc = fmaf(__uint_as_float(wv.y & 0xFFFF0000u), xv.w, acc);
  }
  return acc;
}

struct Args {
  int D, E, F, Fs, k, T;
  float routed_scale;
  const void *router_w;
  int router_f32;
  const float *bias;
  const uint16_t *sg, *su, *sd;
  const uint8_t *experts;
  int64_t expert_bytes, gate_bytes;
  const void *x;
  int x_f32;
  float *logits;
  int32_t *ids;
  float *w;
  int32_t *counts, *offsets, *perm, *pos, *used;
  float *h;   // [P][F] routed activations, perm order
  float *hs;  // [T][Fs]
  unsigned *ctrl;
  float *out;
  int accumulate;
  unsigned *status;
  int n_router, n_sgu, n_rgu, n_down, n_slots;
  int ns;     // ring stages per worker
};

struct Smem {
  int conv_next, conv_done, n_conv;
  int sids[PMAXF];
  float sw[PMAXF];
};

// --------------------------------------------------------------- waits --

__device__ bool wait_ge(const unsigned *p, unsigned target, unsigned *ctrl, unsigned *st) {
  uint64_t t0 = 0;
  unsigned sleep = 64;
  for (unsigned it = 0;; ++it) {
    if (ld_acquire(p) >= target) return true;
    if ((it & 7u) == 7u) {
      if (ld_acquire(ctrl + C_ABORT)) return false;
      const uint64_t now = globaltimer_ns();
      if (!t0) t0 = now;
      else if (now - t0 > WAIT_LIMIT_NS) {
        flag(st, ST_TIMEOUT);
        st_release(ctrl + C_ABORT, 1u);
        return false;
      }
    }
    __nanosleep(sleep);  // back off: thousands of warps may poll the same word
    if (sleep < 1024) sleep *= 2;
  }
}

__device__ bool wait_mbar(uint64_t *bar, uint32_t parity, unsigned *ctrl, unsigned *st) {
  uint64_t t0 = 0;
  for (unsigned it = 0;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;  // non-blocking poll
    if ((it & 255u) == 255u) {
      if (ld_acquire(ctrl + C_ABORT)) return false;
      const uint64_t now = globaltimer_ns();
      if (!t0) t0 = now;
      else if (now - t0 > WAIT_LIMIT_NS) {
        flag(st, ST_TIMEOUT);
        st_release(ctrl + C_ABORT, 1u);
        return false;
      }
    }
    __nanosleep(32);
  }
}

// Warp-uniform bounded wait on a flag (lane 0 waits, the result is broadcast).
__device__ __forceinline__ bool warp_wait_ge(const unsigned *p, unsigned target, unsigned *ctrl,
                                             unsigned *st) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_ge(p, target, ctrl, st) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ------------------------------------------------------------ task plan --

__device__ __forceinline__ int nb_of(int in_dim) { return (in_dim + QK - 1) / QK; }

// Tasks from the first routed gate/up group on need the route.
__device__ __forceinline__ bool routed(const Args &a, int i) { return i >= a.n_router + a.n_sgu; }

// ---------------------------------------------------------------- kernel --

// The route, cached in the registers of every warp once it is known
// (P <= 32: lane p holds pair p, lane u holds used expert u), so inner loops
// never wait on memory for it.
struct RouteCache {
  int nu;      // experts with tokens
  int perm;    // lane p: perm[p]
  float w;     // lane p: w[p]
  int used;    // lane u: used[u]
  int base;    // lane u: offsets[used[u]]
  int cnt;     // lane u: tokens of used[u]
};

__device__ __forceinline__ RouteCache load_route(const Args &a, int P) {
  const int lane = threadIdx.x & 31;
  RouteCache r;
  r.nu = (int)__ldcg((const int *)(a.ctrl + C_NUSED));
  r.perm = lane < P ? __ldcg(a.perm + lane) : 0;
  r.w = lane < P ? __ldcg(a.w + lane) : 0.f;
  r.used = lane < r.nu ? __ldcg(a.used + lane) : 0;
  r.base = lane < r.nu ? __ldcg(a.offsets + r.used) : 0;
  r.cnt = lane < r.nu ? __ldcg(a.offsets + r.used + 1) - r.base : 0;
  return r;
}

__device__ __forceinline__ int shfl(int v, int l) { return __shfl_sync(0xffffffffu, v, l); }
__device__ __forceinline__ float shflf(float v, int l) { return __shfl_sync(0xffffffffu, v, l); }

template <int SPL_D, int SPL_F>
__global__ void __launch_bounds__(NTHREADS, 1) fused_decode_kernel(const Args a) {
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.ns;
  uint8_t *ring = dsm_raw + (size_t)warp * NS * SB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(dsm_raw + (size_t)NW * NS * SB) + warp * NS;
  Smem &sm = *reinterpret_cast<Smem *>(dsm_raw + (size_t)NW * NS * SB + NW * NS * 8);
  const int nsb_d = a.D / 16, nsb_f = a.F / 16, nb_d = a.D / QK, nb_f = a.F / QK;
  const int P = a.T * a.k;
  const int xw = 9 * nsb_d + nb_d, hw = 9 * nsb_f + nb_f;  // words per digit set
  uint32_t *xpl = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(&sm) + ((sizeof(Smem) + 63) & ~63));
  uint32_t *hpl = xpl + a.T * xw;                            // [P] sets, perm order
  float *hs_s = reinterpret_cast<float *>(hpl + P * hw);      // [T][Fs]
  auto xplanes = [&](int t) { return xpl + t * xw; };
  auto xsteps = [&](int t) { return reinterpret_cast<float *>(xpl + t * xw + 9 * nsb_d); };
  auto hplanes = [&](int q) { return hpl + q * hw; };
  auto hsteps = [&](int q) { return reinterpret_cast<float *>(hpl + q * hw + 9 * nsb_f); };
  unsigned *ctrl = a.ctrl, *st = a.status;

  if (lane == 0)
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
  if (threadIdx.x == 0) {
    sm.conv_next = sm.conv_done = 0;
    sm.n_conv = (P * nb_f + 1) / 2 + (a.Fs > 0 ? (a.T * a.Fs + 127) / 128 : 0);
  }
  fence_mbar_init();
  // the tokens' activations in fixed point; each warp converts two blocks at a time
  for (int u = warp; u < (a.T * nb_d + 1) / 2; u += NW) {
    const int bi = 2 * u + (lane >> 4);  // (token, block) index
    const int t = min(bi, a.T * nb_d - 1) / nb_d, b = min(bi, a.T * nb_d - 1) % nb_d;
    float v[16];
    const int64_t e0 = (int64_t)t * a.D + QK * b + 16 * (lane & 15);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = a.x_f32 ? __ldg((const float *)a.x + e0 + j) : bf16_to_f32(__ldg((const uint16_t *)a.x + e0 + j));
    digitize_block<SPL_D>(v, b, xplanes(t), xsteps(t), nsb_d);  // a clamped duplicate rewrites equal values
  }
  __syncthreads();

  const int n_tasks = a.n_router + a.n_sgu + a.n_rgu + a.n_down;
  // tasks are dealt across CTAs first, so every phase is spread over all SMs
  const int gw = warp * gridDim.x + blockIdx.x, nwork = gridDim.x * NW;
  const int groups = a.F / RG;
  const int er = nb_of(a.F) * QB, per = SB / er;            // expert down rows per chunk
  const int sdc = a.Fs > 0 ? (2 * a.Fs + SB - 1) / SB : 0;  // shared down chunks
  // issue cursor (task, chunk) runs ahead of the consume cursor by < NS chunks
  int it_i = gw, it_c = 0, it_kind = -1, it_a = 0, it_b = 0, it_n = 0;
  bool it_have = false;
  int issued = 0, consumed = 0;
  bool ready_seen = false, prologue_done = false, ok = true;
  RouteCache rc{0, 0, 0.f, 0, 0, 0};

  auto route_ready = [&]() -> bool {
    if (!ready_seen) {
      int r = 0;
      if (lane == 0) r = ld_acquire(ctrl + C_READY) != 0;
      if (shfl(r, 0)) {
        __threadfence();
        rc = load_route(a, P);
        ready_seen = true;
      }
    }
    return ready_seen;
  };
  auto wait_route = [&]() -> bool {
    if (route_ready()) return true;
    if (!warp_wait_ge(ctrl + C_READY, 1u, ctrl, st)) return false;
    return route_ready();
  };
  // task i -> (kind, a, b, chunks); needs the route for routed tasks
  auto describe = [&](int i, int &kind, int &ta, int &tb, int &n) {
    kind = -1; ta = tb = n = 0;
    if (i < a.n_router) {
      kind = K_ROUTER; ta = i; n = (a.D * (a.router_f32 ? 4 : 2) + SB - 1) / SB;
      return;
    }
    i -= a.n_router;
    if (i < a.n_sgu) { kind = K_SGU; ta = i; n = 2 * ((2 * a.D + SB - 1) / SB); return; }
    i -= a.n_sgu;
    if (i < a.n_rgu) {
      const int slot = i / groups;
      if (slot >= rc.nu) return;
      kind = K_RGU; ta = shfl(rc.used, slot); tb = slot * groups + i % groups; n = RG;
      return;
    }
    i -= a.n_rgu;
    kind = K_DOWN; ta = i; n = sdc + (rc.nu + per - 1) / per;
  };
  // issue as many chunks as the ring allows; block on the route only when
  // nothing is in flight
  auto fill = [&]() {
    while (ok && issued - consumed < NS) {
      if (!it_have) {
        if (it_i >= n_tasks) return;
        if (routed(a, it_i) && !route_ready()) {
          if (issued > consumed) return;
          if (!wait_route()) { ok = false; return; }
        }
        describe(it_i, it_kind, it_a, it_b, it_n);
        if (it_kind < 0 || it_n == 0) { it_i += nwork; continue; }
        it_have = true;
        it_c = 0;
      }
      const int s = issued % NS;
      uint8_t *stage = ring + s * SB;
      // expert ids a down chunk needs (gathered by every lane)
      int ex[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      int nex = 0;
      if (it_kind == K_DOWN && it_c >= sdc) {
        const int u0 = (it_c - sdc) * per;
        nex = min(rc.nu - u0, per);
#pragma unroll
        for (int v = 0; v < 8; ++v) ex[v] = shfl(rc.used, min(u0 + v, 31));
      }
      if (lane == 0) {
        fence_proxy_async();  // earlier reads of this stage by the warp come first
        if (it_kind == K_ROUTER) {
          const int rb = a.D * (a.router_f32 ? 4 : 2);
          const int off = it_c * SB, n = min(SB, rb - off);
          mbar_arrive_expect_tx(&bars[s], (uint32_t)n);
          bulk_g2s(stage, (const char *)a.router_w + (int64_t)it_a * rb + off, (uint32_t)n, &bars[s]);
        } else if (it_kind == K_SGU) {
          const int pr = (2 * a.D + SB - 1) / SB;
          const uint16_t *row = (it_c < pr ? a.sg : a.su) + (int64_t)it_a * a.D;
          const int off = (it_c % pr) * SB, n = min(SB, 2 * a.D - off);
          mbar_arrive_expect_tx(&bars[s], (uint32_t)n);
          bulk_g2s(stage, (const char *)row + off, (uint32_t)n, &bars[s]);
        } else if (it_kind == K_RGU) {
          const int rb = nb_of(a.D) * QB;
          const int f = (it_b % groups) * RG + it_c;
          const uint8_t *blob = a.experts + (int64_t)it_a * a.expert_bytes;
          mbar_arrive_expect_tx(&bars[s], 2u * rb);
          bulk_g2s(stage, blob + (int64_t)f * rb, (uint32_t)rb, &bars[s]);
          bulk_g2s(stage + rb, blob + a.gate_bytes + (int64_t)f * rb, (uint32_t)rb, &bars[s]);
        } else if (it_c < sdc) {
          const int off = it_c * SB, n = min(SB, 2 * a.Fs - off);
          mbar_arrive_expect_tx(&bars[s], (uint32_t)n);
          bulk_g2s(stage, (const char *)(a.sd + (int64_t)it_a * a.Fs) + off, (uint32_t)n, &bars[s]);
        } else {
          mbar_arrive_expect_tx(&bars[s], (uint32_t)(nex * er));
          for (int v = 0; v < nex; ++v)
            bulk_g2s(stage + v * er,
                     a.experts + (int64_t)ex[v] * a.expert_bytes + 2 * a.gate_bytes + (int64_t)it_a * er,
                     (uint32_t)er, &bars[s]);
        }
      }
      __syncwarp();
      ++issued;
      if (++it_c == it_n) { it_have = false; it_i += nwork; }
    }
  };
  auto wait_chunk = [&]() -> const uint8_t * {
    const int s = consumed % NS;
    const uint32_t par = (uint32_t)((consumed / NS) & 1);
    int r = 1;
    if (lane == 0) r = wait_mbar(&bars[s], par, ctrl, st) ? 1 : 0;
    if (!shfl(r, 0)) { ok = false; return nullptr; }
    while (!mbar_test_wait(&bars[s], par)) {}  // already complete: every lane observes it
    return ring + s * SB;
  };

  for (int ti = gw; ti < n_tasks && ok; ti += nwork) {
    fill();
    if (!ok) break;
    if (routed(a, ti) && !wait_route()) break;
    int kind, ta, tb, nch;
    describe(ti, kind, ta, tb, nch);
    if (kind < 0 || nch == 0) continue;

    if (kind == K_ROUTER) {
      float acc[TMAXF] = {};
      const int rb = a.D * (a.router_f32 ? 4 : 2), esz = a.router_f32 ? 4 : 2;
      for (int c = 0; c < nch; ++c) {
        fill();
        const uint8_t *buf = wait_chunk();
        if (!buf) break;
        const int off = c * SB, n = min(SB, rb - off) / esz, e0 = off / esz;
        for (int tt = 0; tt < a.T; ++tt) {
          const void *xv = a.x_f32 ? (const void *)((const float *)a.x + (int64_t)tt * a.D + e0)
                                   : (const void *)((const uint16_t *)a.x + (int64_t)tt * a.D + e0);
          acc[tt] += dense_dot(buf, a.router_f32, n, xv, a.x_f32 ? 1 : 0);
        }
        __syncwarp();
        ++consumed;
      }
      if (!ok) break;
      const float bias = a.bias ? a.bias[ta] : 0.f;
      for (int tt = 0; tt < a.T; ++tt) {
        const float v = warp_sum(acc[tt]);
        if (lane == 0) a.logits[(int64_t)tt * a.E + ta] = v + bias;
      }
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = atom_add_release(ctrl + C_ROUTER, 1u) == (unsigned)a.n_router - 1u;
      }
      if (shfl(last, 0)) {
        // this warp computes the selection and the route for every token
        __threadfence();
        for (int tt = 0; tt < a.T; ++tt) {
          const float *L = a.logits + (int64_t)tt * a.E;
          float lv[32];  // this lane's logits (E <= 1024), read once
#pragma unroll
          for (int ii = 0; ii < 32; ++ii) lv[ii] = lane + 32 * ii < a.E ? __ldcg(L + lane + 32 * ii) : -INFINITY;
          uint32_t taken = 0;
          float m0 = 0.f;
          for (int j = 0; j < a.k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
              const int e = lane + 32 * ii;
              if (e < a.E && !(taken & (1u << ii)) && (lv[ii] > bv || (lv[ii] == bv && e < bi))) {
                bv = lv[ii];
                bi = e;
              }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
              const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
              if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (bi < 0 || bi >= a.E) { if (lane == 0) flag(st, ST_BAD_ID); bi = 0; }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (j == 0) m0 = bv;
            if (lane == 0) { sm.sids[tt * a.k + j] = bi; sm.sw[tt * a.k + j] = bv; }
          }
          __syncwarp();
          if (lane == 0) {
            float den = 0.f;
            for (int j = 0; j < a.k; ++j) den += __expf(sm.sw[tt * a.k + j] - m0);
            for (int j = 0; j < a.k; ++j) {
              const int p = tt * a.k + j;
              a.ids[p] = sm.sids[p];
              a.w[p] = a.routed_scale * (__expf(sm.sw[p] - m0) / den);
            }
          }
          __syncwarp();
        }
        // stable route: pair p goes to #(smaller expert, or same expert and smaller p)
        int nu = 0;
        for (int p = lane; p < P; p += 32) {
          const int e = sm.sids[p];
          int rank = 0, first = 1, ui = 0;
          for (int q = 0; q < P; ++q) {
            const int eq = sm.sids[q];
            rank += (eq < e) || (eq == e && q < p);
            if (eq == e && q < p) first = 0;
          }
          if (first) {
            for (int q = 0; q < P; ++q) {  // distinct experts below e
              const int eq = sm.sids[q];
              bool fq = eq < e;
              for (int q2 = 0; q2 < q && fq; ++q2) fq = sm.sids[q2] != eq;
              ui += fq;
            }
            a.used[ui] = e;
          }
          a.perm[rank] = p;
          a.pos[p] = rank;
          nu += first;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) nu += __shfl_xor_sync(0xffffffffu, nu, o);
        for (int e = lane; e <= a.E; e += 32) {
          int lt = 0, eqc = 0;
          for (int q = 0; q < P; ++q) { lt += sm.sids[q] < e; eqc += sm.sids[q] == e; }
          a.offsets[e] = lt;
          if (e < a.E) a.counts[e] = eqc;
        }
        if (lane == 0) {
          a.used[a.E] = nu;
          ctrl[C_NUSED] = (unsigned)nu;
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(ctrl + C_READY, 1u);
      }
    } else if (kind == K_SGU) {
      float g[TMAXF] = {}, u[TMAXF] = {};
      const int pr = nch / 2;
      for (int c = 0; c < nch; ++c) {
        fill();
        const uint8_t *buf = wait_chunk();
        if (!buf) break;
        const int cc = c % pr, e0 = cc * SB / 2, n = min(SB, 2 * a.D - cc * SB) / 2;
        for (int tt = 0; tt < a.T; ++tt) {
          const void *xv = a.x_f32 ? (const void *)((const float *)a.x + (int64_t)tt * a.D + e0)
                                   : (const void *)((const uint16_t *)a.x + (int64_t)tt * a.D + e0);
          const float v = dense_dot(buf, false, n, xv, a.x_f32 ? 1 : 0);
          if (c < pr) g[tt] += v; else u[tt] += v;
        }
        __syncwarp();
        ++consumed;
      }
      if (!ok) break;
      for (int tt = 0; tt < a.T; ++tt) {
        const float gs = warp_sum(g[tt]), us = warp_sum(u[tt]);
        if (lane == 0) a.hs[(int64_t)tt * a.Fs + ta] = silu(gs) * us;
      }
      if (lane == 0) { __threadfence(); atom_add_release(ctrl + C_GU, 1u); }
    } else if (kind == K_RGU) {
      const int slot = tb / groups, grp = tb % groups;
      const int base = shfl(rc.base, slot), n = shfl(rc.cnt, slot);
      const int rb = nb_of(a.D) * QB;
      for (int c = 0; c < RG; ++c) {
        fill();
        const uint8_t *buf = wait_chunk();
        if (!buf) break;
        const int f = grp * RG + c;
        for (int j = 0; j < n; ++j) {
          const int tt = shfl(rc.perm, base + j) / a.k;
          const float gs = warp_sum(q2k_dot<SPL_D>(buf, xplanes(tt), xsteps(tt), nsb_d));
          const float us = warp_sum(q2k_dot<SPL_D>(buf + rb, xplanes(tt), xsteps(tt), nsb_d));
          if (lane == 0) a.h[(int64_t)(base + j) * a.F + f] = silu(gs) * us;
        }
        __syncwarp();
        ++consumed;
      }
      if (!ok) break;
      if (lane == 0) { __threadfence(); atom_add_release(ctrl + C_GU, 1u); }
    } else {
      // ------------------------------------------------------------ down row
      if (!prologue_done) {
        // every gate/up result exists; turn them into shared-memory operands
        // once per CTA, shared out among the workers that arrive
        const unsigned target = (unsigned)(a.n_sgu + rc.nu * groups);
        if (!warp_wait_ge(ctrl + C_GU, target, ctrl, st)) break;
        __threadfence();
        const int nhu = (P * nb_f + 1) / 2;  // units of two (pair, block) conversions
        for (;;) {
          int unit = 0;
          if (lane == 0) unit = atomicAdd(&sm.conv_next, 1);
          unit = shfl(unit, 0);
          if (unit >= sm.n_conv) break;
          if (unit < nhu) {
            const int bi = min(2 * unit + (lane >> 4), P * nb_f - 1);  // (pair position, block)
            const int q = bi / nb_f, b = bi % nb_f;
            float v[16];
            const float4 *src = reinterpret_cast<const float4 *>(a.h + (int64_t)q * a.F + QK * b + 16 * (lane & 15));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 f4 = __ldcg(src + j);
              v[4 * j] = f4.x; v[4 * j + 1] = f4.y; v[4 * j + 2] = f4.z; v[4 * j + 3] = f4.w;
            }
            digitize_block<SPL_F>(v, b, hplanes(q), hsteps(q), nsb_f);
          } else {
            const int i4 = (unit - nhu) * 32 + lane;  // float4 of hs
            if (i4 < a.T * a.Fs / 4)
              reinterpret_cast<float4 *>(hs_s)[i4] = __ldcg(reinterpret_cast<const float4 *>(a.hs) + i4);
          }
          __syncwarp();
          if (lane == 0) { __threadfence_block(); atomicAdd(&sm.conv_done, 1); }
        }
        // wait (bounded) until every unit of this CTA is converted
        int r = 1;
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          while (atomicAdd(&sm.conv_done, 0) < sm.n_conv) {
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
              flag(st, ST_TIMEOUT);
              st_release(ctrl + C_ABORT, 1u);
              r = 0;
              break;
            }
            __nanosleep(256);
          }
          __threadfence_block();
        }
        if (!shfl(r, 0)) break;
        __syncwarp();
        prologue_done = true;
      }
      const int d = ta;
      float ys[TMAXF] = {};
      float yreg = 0.f;  // lane p: y of pair p for this output row
      for (int c = 0; c < nch; ++c) {
        fill();
        const uint8_t *buf = wait_chunk();
        if (!buf) break;
        if (c < sdc) {
          const int e0 = c * SB / 2, n = min(SB, 2 * a.Fs - c * SB) / 2;
          for (int tt = 0; tt < a.T; ++tt) ys[tt] += dense_dot_s(buf, n, hs_s + (int64_t)tt * a.Fs + e0);
        } else {
          const int u0 = (c - sdc) * per, u1 = min(rc.nu, u0 + per);
          for (int u = u0; u < u1; ++u) {
            const int base = shfl(rc.base, u), n = shfl(rc.cnt, u);
            for (int j = 0; j < n; ++j) {
              const float y = warp_sum(q2k_dot<SPL_F>(buf + (u - u0) * er, hplanes(base + j),
                                                      hsteps(base + j), nsb_f));
              if (lane == shfl(rc.perm, base + j)) yreg = y;
            }
          }
        }
        __syncwarp();
        ++consumed;
      }
      if (!ok) break;
      for (int tt = 0; tt < a.T; ++tt) {
        float acc = warp_sum(ys[tt]);  // y_shared (0 without a shared expert)
        for (int j = 0; j < a.k; ++j) {
          const int p = tt * a.k + j;
          acc = fmaf(shflf(rc.w, p), shflf(yreg, p), acc);
        }
        if (lane == 0) {
          float *o = a.out + (int64_t)tt * a.D + d;
          *o = a.accumulate ? *o + acc : acc;
        }
      }
      __syncwarp();
    }
  }
  // never leave while a bulk copy into this warp's ring may still be landing
  if (lane == 0) {
    for (int j = max(consumed, issued - NS); j < issued; ++j) {
      const int s = j % NS;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars[s], (uint32_t)((j / NS) & 1))) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) { flag(st, ST_TIMEOUT); break; }
      }
    }
  }
  __syncwarp();
}

size_t smem_bytes(int T, int k, int D, int F, int Fs, int ns) {
  const int P = T * k;
  return (size_t)NW * ns * SB + NW * ns * 8 + ((sizeof(Smem) + 63) & ~(size_t)63) +
         4 * ((size_t)T * (9 * (D / 16) + D / QK) + (size_t)P * (9 * (F / 16) + F / QK)) +
         sizeof(float) * (size_t)T * Fs;
}

}  // namespace

// (n_embd, n_ff) block counts with an instantiated kernel
static bool fused_shape_ok(int nb_d, int nb_f) {
  return (nb_d == 16 && nb_f == 8) || (nb_d == 4 && nb_f == 4) || (nb_d == 8 && nb_f == 8) ||
         (nb_d == 16 && nb_f == 16);
}

bool fused_decode_supported(const Shape &sh, int64_t T) {
  if (T < 1 || T > TMAXF || (int64_t)T * sh.k > PMAXF) return false;
  if (sh.D % QK || sh.F % QK || !fused_shape_ok(sh.D / QK, sh.F / QK)) return false;
  if (2 * (sh.D / QK) * QB > SB || (sh.F / QK) * QB > SB) return false;
  return smem_bytes((int)T, sh.k, sh.D, sh.F, sh.Fs, 2) <= SMEM_LIMIT;
}

cudaError_t launch_decode_fused(const Shape &sh, const ds_moe_weights &W, const void *x,
                                const Work &wk, float *out, bool accumulate, cudaStream_t s) {
  Args a{};
  a.D = sh.D; a.E = sh.E; a.F = sh.F; a.Fs = sh.Fs; a.k = sh.k; a.T = (int)wk.T;
  a.routed_scale = sh.routed_scale;
  a.router_w = W.router_w;
  a.router_f32 = sh.router_dtype == DS_F32;
  a.bias = W.router_bias;
  a.sg = W.shared_gate; a.su = W.shared_up; a.sd = W.shared_down;
  a.experts = W.experts_q2k;
  a.expert_bytes = sh.expert_bytes();
  a.gate_bytes = sh.gate_bytes();
  a.x = x;
  a.x_f32 = sh.x_dtype == DS_F32;
  a.logits = wk.logits; a.ids = wk.ids; a.w = wk.w;
  a.counts = wk.counts; a.offsets = wk.offsets; a.perm = wk.perm; a.pos = wk.pos; a.used = wk.used;
  a.h = wk.h;
  a.hs = wk.hs;
  a.ctrl = wk.ctrl;
  a.out = out;
  a.accumulate = accumulate ? 1 : 0;
  a.status = status_word();
  a.n_router = sh.E;
  a.n_sgu = sh.Fs;
  a.n_slots = (int)std::min<int64_t>(sh.E, wk.T * sh.k);
  a.n_rgu = a.n_slots * (sh.F / RG);
  a.n_down = sh.D;
  a.ns = smem_bytes(a.T, sh.k, sh.D, sh.F, sh.Fs, 3) <= SMEM_LIMIT ? 3 : 2;
  const size_t smem = smem_bytes(a.T, sh.k, sh.D, sh.F, sh.Fs, a.ns);
  const int nb_d = sh.D / QK, nb_f = sh.F / QK;
  const void *kern = nullptr;
  int which = 0;
  if (nb_d == 16 && nb_f == 8) { kern = (const void *)fused_decode_kernel<8, 4>; which = 0; }
  else if (nb_d == 4 && nb_f == 4) { kern = (const void *)fused_decode_kernel<2, 2>; which = 1; }
  else if (nb_d == 8 && nb_f == 8) { kern = (const void *)fused_decode_kernel<4, 4>; which = 2; }
  else if (nb_d == 16 && nb_f == 16) { kern = (const void *)fused_decode_kernel<8, 8>; which = 3; }
  else return cudaErrorInvalidValue;
  static bool attr[4] = {};
  if (!attr[which]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    attr[which] = true;
  }
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  cudaError_t e = cudaMemsetAsync(wk.ctrl, 0, 64, s);
  if (e != cudaSuccess) return e;
  void *params[] = {&a};
  return cudaLaunchCooperativeKernel(kern, dim3(sms), dim3(NTHREADS), params, smem, s);
}

}  // namespace dsm
