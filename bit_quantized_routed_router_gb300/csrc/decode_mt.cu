// Batched decode: the layer for 4..16 tokens with every used expert's weights
// read once.
//
// What it computes is the layer of "Understanding Dwarf Star" 5.3.2 / 5.3.7
// (router -> top-k -> gate/up -> SiLU(gate) * up -> down -> weighted sum)
// with the always-active shared expert of 5.3.4 and the routed weights read as
// Q2_K blocks (3.3.3), dequantised on the fly (2.8.1-2.8.2).  The pages batch
// decode rows of several sessions into one pass over the experts ("DwarfStar
// Native Inference Engine", micro-batched generation); here a batch of T
// tokens is one pass.
//
// After the router logits (router_small_kernel), four kernels chained with
// programmatic dependent launch:
//
//   mt_gu_kernel  every block selects the top-k of all T tokens and builds the
//                 route in shared memory (block 0 publishes it); a copy warp
//                 streams weight tiles through a ring of shared-memory stages
//                 with bulk-tensor copies; eight warps consume them:
//                   shared expert  128 bf16 rows x 64 K per tile with the
//                                  tokens' 64 K of x, on the tensor cores
//                                  (mma.sync m16n8k16 bf16, fp32 accumulators:
//                                  products exact), partial sums per 1024 K;
//                   routed expert  32 Q2_K row pairs (gate, up) x 1024 K per
//                                  tile; exact integer row dots (dp4a) with the
//                                  16-bit fixed-point activation planes of the
//                                  expert's tokens, held in shared memory.
//                 Each block owns one K slice of n_embd for the routed rows (so
//                 that the planes of all T tokens fit); it writes partial gate
//                 and up sums per slice.  Routed tiles are dealt round-robin,
//                 so a hot expert's tiles spread over all blocks.
//   mt_h_kernel   h = SiLU(sum of gate slices) * (sum of up slices), turned
//                 into fixed-point planes per routed pair, and the shared
//                 activations split into bf16 hi + lo (hs = hi + lo to 2^-17).
//   mt_dn_kernel  down rows: routed tiles of 64 Q2_K rows x 1024 K with the
//                 planes of the expert's pairs (copied into shared memory per
//                 expert, so a block takes a contiguous range of tiles whose
//                 bytes and token work add up to its share); shared tiles of
//                 128 bf16 rows x 64 K with hs hi and lo on the tensor cores.
//                 Partial sums per K slice of n_ff and per 1024 K of the shared
//                 width.
//   mt_combine    out = y_shared + sum_j w_j y_j (pair order j), the K slices
//                 of each term added in a fixed order.
//
// Every reduction has a fixed order, so the result does not depend on
// scheduling.  Every wait is bounded; an expired wait sets ST_TIMEOUT and the
// kernel winds down.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "qrows.cuh"
#include "select.cuh"

namespace dsm {
namespace {

constexpr int MT_CONS = 8;                      // consumer warps
constexpr int MT_THREADS = MT_CONS * 32;       // lane 0 of the last warp also issues the copies
constexpr int MT_NC = MT_CONS * 32;             // consumer threads
constexpr int MT_NS = 4;                        // ring stages
constexpr uint32_t MT_STAGE = 24576;            // bytes per stage (a multiple of 1024)
constexpr int MT_CHUNK = 1024;                  // activation elements per plane chunk (4 blocks)
constexpr int MT_TCH = 32;                      // plane chunks a block holds (tokens or pairs x chunks)
constexpr int MT_MAXT = 32;                     // tokens per call
constexpr int MT_MAXP = 512;                    // token-expert pairs per call
constexpr int MT_SH_ROWS = 128;                 // shared-expert rows per tile (16 per warp)
constexpr int MT_BOX_K = 64;                    // K of a shared-expert tile (one 128-byte row)
constexpr uint32_t MT_SH_BOX = MT_SH_ROWS * 128;  // bytes of a shared-expert weight tile
constexpr uint64_t MT_LIMIT_NS = 2000000000ull;
constexpr size_t MT_SMEM_LIMIT = 227 * 1024;

// Row format of the routed experts for a 1024-element chunk: Q2_K rows with
// two sub-blocks per lane (four blocks over 32 lanes).
using RQ = Q2Rows<2>;
constexpr int MT_CB = 4 * QB;                              // bytes of one row's chunk (336)
constexpr int MT_CHW = RQ::NPL * (MT_CHUNK / RQ::SUB) + 4;  // plane words per chunk (580)
constexpr int MT_GU_RP = 4;                                // routed gate/up row pairs per warp
constexpr int MT_GU_NR = MT_CONS * MT_GU_RP;               // row pairs per gate/up tile (32)
constexpr int MT_DN_R = 8;                                 // routed down rows per warp
constexpr int MT_DN_NR = MT_CONS * MT_DN_R;                // rows per down tile (64)
static_assert(2 * MT_GU_NR * MT_CB <= (int)MT_STAGE && MT_DN_NR * MT_CB <= (int)MT_STAGE, "routed tile");
static_assert(MT_SH_BOX + 2 * MT_MAXT * 128 <= MT_STAGE, "shared tile");
static_assert(2 * MT_GU_RP <= 8 && 32 % (2 * MT_GU_RP) == 0 && MT_DN_R <= 8 && 32 % MT_DN_R == 0,
              "values per warp: at most eight, spread evenly over the lanes");

struct MtArgs {
  int D, E, F, Fs, k, T, T8, P;
  int KS, KSd;              // K slices of n_embd (gate/up) and of n_ff, n_ff_shared (down)
  float routed_scale, logit_scale;
  const float *unbias;      // the router bias when it steers the selection only
  const uint8_t *experts;
  int64_t expert_bytes, gate_bytes;
  const uint16_t *x;        // [T][D] bf16
  const float *logits;      // [T][E]
  int32_t *ids;             // route, published by block 0 of the gate/up kernel
  float *w;
  int32_t *counts, *offsets, *perm, *pos, *used;
  unsigned *ctrl;
  float *gp, *up;           // [KS][P][F] partial routed gate / up
  float *gs, *us;           // [D / 1024][T][Fs] partial shared gate / up
  uint32_t *hpl;            // [P][F / 1024][MT_CHW] planes of h
  uint16_t *hs_hi, *hs_lo;  // [T][Fs] shared activations, bf16 hi + lo
  float *y;                 // [KSd][P][D] partial routed down
  float *ys;                // [Fs / 1024][T][D] partial shared down
  float *out;
  int accumulate;
  unsigned *status;
};

enum { C_NUSED = 1 };  // control word: experts with tokens (written with the route)

struct MtShared {
  uint64_t full[MT_NS], empty[MT_NS];
  uint64_t planes_full, planes_empty;  // down kernel: the pair planes of the current expert
  int4 desc[MT_NS];  // the tile in each stage
  int route_ready;
  int abort_;
  int nu;
};

__device__ __forceinline__ int vld(const int *p) { return *(volatile const int *)p; }

__device__ bool mt_wait(uint64_t *bar, uint32_t par, MtShared &S, unsigned *status) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, par, 20000u)) {
    if (vld(&S.abort_)) return false;
    if (globaltimer_ns() - t0 > MT_LIMIT_NS) {
      flag(status, ST_TIMEOUT);
      *(volatile int *)&S.abort_ = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t r[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

// D += A B: A 16 x 16 bf16 (row-major fragment), B 16 x 8 bf16, fp32 D.
__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], const uint32_t b[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Address of 16-byte chunk c of row r in a tile of 128-byte rows stored by a
// bulk-tensor copy in the 128-byte swizzle (chunk c of row r at c ^ (r mod 8)).
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ int count_of(int n, int j, int G) { return n > j ? (n - j + G - 1) / G : 0; }

// Round-robin deal of a slice group's routed items (block j of Gq blocks of
// slice q; slices interleave the grid's G blocks, block b = q + KS j): the
// deal starts after the blocks that hold one more shared-expert item than the
// rest (S shared items dealt round-robin over all G blocks first).
__device__ __forceinline__ int rr_first(int j, int q, int KS, int Gq, int S, int G) {
  const int extra = S % G;
  const int off = extra > q ? (extra - q + KS - 1) / KS : 0;
  return ((j - off) % Gq + Gq) % Gq;
}

// Contiguous routed ranges for the down kernel (items expert-major, NG per
// expert, cost w_u = NCqd (2 + n_u) each: a tile's bytes count two, each
// token's dots one), balanced over the Gq blocks of a slice group together
// with each block's shared-expert items (cost c_sh each).  Block j takes the
// items whose cost midpoint lies in [B_j, B_{j+1}), B_j the running maximum of
// j * total / Gq - (shared cost of blocks < j); every block computes the same
// boundaries, so the ranges partition the items.
__device__ int cost_boundary(int j, int Gq, int q, int KS, int G, int S, int c_sh, int nu, const int32_t *cnt,
                             int NCqd, int NG) {
  int64_t rt_total = 0;
  for (int u = 0; u < nu; ++u) rt_total += (int64_t)NG * NCqd * (2 + cnt[u]);
  int64_t sh_total = 0;
  for (int jj = 0; jj < Gq; ++jj) sh_total += (int64_t)count_of(S, q + KS * jj, G) * c_sh;
  const int64_t total = rt_total + sh_total;
  // 2 Gq B_j, as a running maximum
  int64_t tj = 0, sh_before = 0;
  for (int jj = 0; jj <= j && jj < Gq; ++jj) {
    const int64_t t = 2 * ((int64_t)jj * total - (int64_t)Gq * sh_before);
    tj = t > tj ? t : tj;
    sh_before += (int64_t)count_of(S, q + KS * jj, G) * c_sh;
  }
  if (j >= Gq) return nu * NG;
  int64_t c0 = 0;  // cost before expert u
  for (int u = 0; u < nu; ++u) {
    const int64_t w = (int64_t)NCqd * (2 + cnt[u]);
    // first item i with 2 Gq (c0 + i w) + Gq w >= tj
    const int64_t num = tj - (int64_t)Gq * w - 2 * (int64_t)Gq * c0, den = 2 * (int64_t)Gq * w;
    const int64_t i = num <= 0 ? 0 : (num + den - 1) / den;
    if (i < NG) return u * NG + (int)i;
    c0 += (int64_t)NG * w;
  }
  return nu * NG;
}

// 16 bf16 rows of a shared-expert tile (warp w: rows 16 w ..) times the
// tokens: per 16-K step the A fragment, then the B fragment of every token
// group (T8 / 8 of them) from one or two token tiles (tok_lo adds a low part
// of the activations), accumulated into c.  The stage is released after the
// last fragment load.
__device__ __forceinline__ void shared_tile_mma(uint32_t wtile, uint32_t tok_hi, uint32_t tok_lo, bool two, int T8,
                                                float c[MT_MAXT / 8][4], uint64_t *empty) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= MT_SH_ROWS / 16) {  // 16 rows per warp: the other warps only release the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);
    return;
  }
  const int mi = lane >> 3, ra = 16 * warp + (mi & 1) * 8 + (lane & 7);
  const int rb = lane & 7, cb = (lane >> 3) & 1;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    uint32_t a[4];
    ldsm_x4(sw_addr(wtile, ra, 2 * ks + (mi >> 1)), a);
#pragma unroll
    for (int tg = 0; tg < MT_MAXT / 8; ++tg)
      if (tg * 8 < T8) {
        uint32_t b[2];
        ldsm_x2(sw_addr(tok_hi, tg * 8 + rb, 2 * ks + cb), b);
        mma_bf16(c[tg], a, b);
        if (two) {
          ldsm_x2(sw_addr(tok_lo, tg * 8 + rb, 2 * ks + cb), b);
          mma_bf16(c[tg], a, b);
        }
      }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);
}

// Stores the shared-tile accumulators: rows row0 + 16 w + g (+ 8), tokens
// 8 tg + 2 t (+ 1) -> dst[t * ld + row] for t < T.
__device__ __forceinline__ void store_shared_acc(const float c[MT_MAXT / 8][4], float *dst, int64_t ld, int row0,
                                                 int T) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t2 = 2 * (lane & 3);
  if (warp >= MT_SH_ROWS / 16) return;
  const int r = row0 + 16 * warp + g;
#pragma unroll
  for (int tg = 0; tg < MT_MAXT / 8; ++tg) {
    const int t = 8 * tg + t2;
    if (t < T) { dst[(int64_t)t * ld + r] = c[tg][0]; dst[(int64_t)t * ld + r + 8] = c[tg][2]; }
    if (t + 1 < T) { dst[(int64_t)(t + 1) * ld + r] = c[tg][1]; dst[(int64_t)(t + 1) * ld + r + 8] = c[tg][3]; }
  }
}

// ================================================================ gate/up ==

struct GuLayout {
  size_t shared_off, planes_off, route_off, acc_off, total;
};

__host__ __device__ inline size_t al128(size_t v) { return (v + 127) & ~(size_t)127; }

__host__ __device__ inline GuLayout gu_layout(int T, int NCq, int E, int P) {
  GuLayout L;
  L.shared_off = (size_t)MT_NS * MT_STAGE;
  L.planes_off = L.shared_off + al128(sizeof(MtShared));
  L.route_off = L.planes_off + al128((size_t)T * NCq * MT_CHW * 4);
  L.acc_off = L.route_off + al128((size_t)(5 * P + 3 * E + 1) * 4);
  L.total = L.acc_off + (NCq > 1 ? (size_t)MT_CONS * T * 8 * 4 : 0);
  return L;
}

__global__ void __launch_bounds__(MT_THREADS, 1)
    mt_gu_kernel(const MtArgs a, const __grid_constant__ CUtensorMap m_rgu, const __grid_constant__ CUtensorMap m_sg,
                 const __grid_constant__ CUtensorMap m_su, const __grid_constant__ CUtensorMap m_x) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int T = a.T, E = a.E, k = a.k, P = a.P, F = a.F, Fs = a.Fs;
  const int G = gridDim.x, b = blockIdx.x;
  const int NCd = a.D / MT_CHUNK, NCq = NCd / a.KS;
  const int q = b % a.KS, bq = b / a.KS;
  const int Gq = (G - q + a.KS - 1) / a.KS;  // blocks of this slice
  const GuLayout L = gu_layout(T, NCq, E, P);
  uint8_t *stages = smem;
  MtShared &S = *reinterpret_cast<MtShared *>(smem + L.shared_off);
  uint32_t *xpl = reinterpret_cast<uint32_t *>(smem + L.planes_off);
  int32_t *s_ids = reinterpret_cast<int32_t *>(smem + L.route_off);
  float *s_w = reinterpret_cast<float *>(s_ids + P);
  int32_t *s_pos = s_ids + 2 * P, *s_tok = s_ids + 3 * P, *s_perm = s_ids + 4 * P;
  int32_t *s_cnt = s_ids + 5 * P, *s_off = s_cnt + E, *s_used = s_off + E + 1;
  float *s_acc = reinterpret_cast<float *>(smem + L.acc_off);

  // shared-expert items: (128-row group of gate or up, 1024-wide chunk of
  // n_embd), dealt round-robin over all blocks; routed items: (expert slot,
  // 32 row pairs), the chunks of this block's slice each, dealt round-robin
  // over the slice's blocks
  const int n_sh_groups = 2 * (Fs / MT_SH_ROWS);
  const int S_items = n_sh_groups * NCd;
  const int NB = MT_CHUNK / MT_BOX_K;             // boxes per shared item
  const int n_sh = count_of(S_items, b, G);
  const int NG = F / MT_GU_NR;                    // routed row groups per expert
  const int rr0 = rr_first(bq, q, a.KS, Gq, S_items, G);

  if (tid == 0) {
    for (int i = 0; i < MT_NS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], MT_CONS);
    }
    S.route_ready = 0;
    S.abort_ = 0;
    S.nu = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Lane 0 of the last warp issues the bulk-tensor copies: tile i of this
  // block into stage i mod MT_NS, once every warp has released the tile that
  // was there.  Shared-expert tiles (no route needed) come first.
  const bool producer = warp == MT_CONS - 1 && lane == 0;
  int n_tiles = n_sh * NB;  // routed tiles are added once the route is known
  // the tiles are issued in order: their coordinates advance without divisions
  int p_kb = 0, p_c = b % NCd, p_sg = b / NCd;                   // shared: item b + G m, box kb
  const int p_gd = G / NCd, p_gm = G % NCd;
  int p_cl = 0, p_u = rr0 / max(NG, 1), p_g = rr0 % max(NG, 1);  // routed: item rr0 + Gq r, chunk cl
  const int p_qd = Gq / max(NG, 1), p_qm = Gq % max(NG, 1);
  auto issue = [&](int i) -> bool {
    const int st = i % MT_NS;
    if (i >= MT_NS && !mt_wait(&S.empty[st], ((i / MT_NS) & 1) ^ 1, S, a.status)) return false;
    uint8_t *dst = stages + (size_t)st * MT_STAGE;
    if (i < n_sh * NB) {
      const int kb = p_kb, c = p_c, sg = p_sg;
      if (++p_kb == NB) {
        p_kb = 0;
        p_c += p_gm;
        p_sg += p_gd;
        if (p_c >= NCd) p_c -= NCd, ++p_sg;
      }
      const bool gate = sg < n_sh_groups / 2;
      const int row0 = (gate ? sg : sg - n_sh_groups / 2) * MT_SH_ROWS;
      S.desc[st] = make_int4(0, sg, kb, c);
      mbar_arrive_expect_tx(&S.full[st], MT_SH_BOX + (uint32_t)a.T8 * 128);
      const int kx = c * MT_CHUNK + kb * MT_BOX_K;
      tma2d(dst, gate ? &m_sg : &m_su, kx, row0, &S.full[st]);
      tma2d(dst + MT_SH_BOX, &m_x, kx, 0, &S.full[st]);
    } else {
      const int cl = p_cl, u = p_u, g = p_g, e = s_used[u];
      if (++p_cl == NCq) {
        p_cl = 0;
        p_g += p_qm;
        p_u += p_qd;
        if (p_g >= NG) p_g -= NG, ++p_u;
      }
      S.desc[st] = make_int4(1, u, g, cl);
      mbar_arrive_expect_tx(&S.full[st], 2u * MT_GU_NR * MT_CB);
      const int xw = (q * NCq + cl) * (MT_CB / 4);
      tma3d(dst, &m_rgu, xw, g * MT_GU_NR, e, &S.full[st]);
      tma3d(dst + MT_GU_NR * MT_CB, &m_rgu, xw, F + g * MT_GU_NR, e, &S.full[st]);
    }
    return true;
  };
  int issued = 0;  // (producer lane)
  if (producer) {
    for (const CUtensorMap *m : {&m_rgu, &m_sg, &m_su, &m_x})
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
    while (issued < MT_NS && issued < n_tiles && issue(issued)) ++issued;
  }

  // --------------------------------------------------------- consumers --
  // 1. fixed-point planes of this slice of every token (half a warp per
  //    256-element block)
  {
    const int nblk = T * NCq * 4;
    for (int u0 = warp; u0 < (nblk + 1) / 2; u0 += MT_CONS) {
      const int bi = min(2 * u0 + (lane >> 4), nblk - 1);
      const int t = bi / (NCq * 4), cb = bi % (NCq * 4), cl = cb / 4, bb = cb % 4;
      const uint16_t *src = a.x + (int64_t)t * a.D + (int64_t)(q * NCq + cl) * MT_CHUNK + QK * bb + 16 * (lane & 15);
      const uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(src)), v1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
      float v[16];
      bf16x8(v0, v);
      bf16x8(v1, v + 8);
      uint32_t *pl = xpl + (size_t)(t * NCq + cl) * MT_CHW;
      RQ::digitize(v, bb, pl, reinterpret_cast<float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB);
    }
  }
  // 2. top-k of every token, then the route (counting sort, stable)
  pdl_wait();  // router logits complete and visible
  for (int t = warp; t < T; t += MT_CONS)
    select_token(a.logits + (int64_t)t * E, E, k, a.routed_scale, a.logit_scale, a.unbias, s_ids + t * k,
                 s_w + t * k, a.status);
  for (int e = tid; e < E; e += MT_NC) s_cnt[e] = 0;
  named_bar(1, MT_NC);
  for (int p = tid; p < P; p += MT_NC) {
    int e = s_ids[p];
    if (e < 0 || e >= E) { flag(a.status, ST_BAD_ID); e = 0; s_ids[p] = 0; }
    atomicAdd(&s_cnt[e], 1);
  }
  named_bar(1, MT_NC);
  if (warp == 0) {
    int run = 0, nu = 0;
    for (int b0 = 0; b0 < E; b0 += 32) {
      const int e = b0 + lane;
      const int c = e < E ? s_cnt[e] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) s_off[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
      const unsigned m = __ballot_sync(0xffffffffu, c > 0);
      if (c > 0) s_used[nu + __popc(m & ((1u << lane) - 1u))] = e;
      nu += __popc(m);
    }
    if (lane == 0) { s_off[E] = run; S.nu = nu; }
  }
  named_bar(1, MT_NC);
  for (int p = tid; p < P; p += MT_NC) {
    const int e = s_ids[p];
    int r = 0;
    for (int qq = 0; qq < p; ++qq) r += s_ids[qq] == e;
    const int at = s_off[e] + r;
    s_pos[p] = at;
    s_perm[at] = p;
    s_tok[at] = p / k;
  }
  named_bar(1, MT_NC);
  const int nu = S.nu;
  if (tid == 0) {
    __threadfence_block();
    *(volatile int *)&S.route_ready = 1;
  }
  if (b == 0) {  // publish the route for the next kernels and the debug outputs
    for (int p = tid; p < P; p += MT_NC) {
      a.ids[p] = s_ids[p];
      a.w[p] = s_w[p];
      a.perm[p] = s_perm[p];
      a.pos[p] = s_pos[p];
    }
    for (int e = tid; e <= E; e += MT_NC) {
      a.offsets[e] = s_off[e];
      if (e < E) a.counts[e] = s_cnt[e];
    }
    for (int u = tid; u < nu; u += MT_NC) a.used[u] = s_used[u];
    if (tid == 0) {
      a.used[E] = nu;
      a.ctrl[C_NUSED] = (unsigned)nu;
    }
  }
  // the next kernels wait for this grid to finish before they read anything
  pdl_trigger();

  // 3. the tiles, in the order they are issued
  n_tiles += count_of(nu * NG, rr0, Gq) * NCq;
  if (producer)
    while (issued < MT_NS && issued < n_tiles && issue(issued)) ++issued;
  // after a tile's stage is released: the tile MT_NS places ahead into it
  auto refill = [&](int kq) {
    if (producer && issued == kq + MT_NS && issued < n_tiles && issue(issued)) ++issued;
  };
  float c[MT_MAXT / 8][4];
#pragma unroll
  for (int tg = 0; tg < MT_MAXT / 8; ++tg) c[tg][0] = c[tg][1] = c[tg][2] = c[tg][3] = 0.f;
  const uint32_t stages_u32 = smem_u32(stages);
  for (int kq = 0; kq < n_tiles; ++kq) {
    const int st = kq % MT_NS;
    const bool got = mt_wait(&S.full[st], (kq / MT_NS) & 1, S, a.status);
    if (!got) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      continue;
    }
    const int4 d = S.desc[st];
    const uint32_t sbase = stages_u32 + (uint32_t)st * MT_STAGE;
    if (d.x == 0) {
      // shared expert: 16 rows per warp x the tokens, 64 K per tile
      const int sg = d.y, kb = d.z, cc = d.w;
      shared_tile_mma(sbase, sbase + MT_SH_BOX, 0, false, a.T8, c, &S.empty[st]);
      refill(kq);
      if (kb == NB - 1) {
        const bool gate = sg < n_sh_groups / 2;
        const int row0 = (gate ? sg : sg - n_sh_groups / 2) * MT_SH_ROWS;
        store_shared_acc(c, (gate ? a.gs : a.us) + (int64_t)cc * T * Fs, Fs, row0, T);
#pragma unroll
        for (int tg = 0; tg < MT_MAXT / 8; ++tg) c[tg][0] = c[tg][1] = c[tg][2] = c[tg][3] = 0.f;
      }
      continue;
    }
    // routed expert slot u, row group g, chunk cl of the slice: the warp's
    // four gate rows and four up rows; for three or more tokens with the scales
    // folded into the codes (the same integer sums, fewer instructions per
    // token)
    const int u = d.y, g = d.z, cl = d.w;
    const int e = s_used[u], base = s_off[e], n = s_cnt[e];
    const uint8_t *tile = stages + (size_t)st * MT_STAGE;
    // lane LV i holds value i: the warp's gate rows, then its up rows
    constexpr int LV = 32 / (2 * MT_GU_RP);
    const int vi = lane / LV;
    const int f = g * MT_GU_NR + warp * MT_GU_RP + vi % MT_GU_RP;
    auto emit = [&](int j, float tot) {
      if (lane % LV == 0) {
        if (NCq > 1) {
          float *acc = s_acc + ((size_t)warp * T + j) * 8 + vi;
          tot = cl == 0 ? tot : *acc + tot;
          *acc = tot;
        }
        if (cl == NCq - 1) (vi < MT_GU_RP ? a.gp : a.up)[((int64_t)q * P + base + j) * F + f] = tot;
      }
    };
    auto row_of = [&](int i) {
      return tile + (size_t)(i < MT_GU_RP ? warp * MT_GU_RP + i : MT_GU_NR + warp * MT_GU_RP + i - MT_GU_RP) * MT_CB;
    };
    if (n <= 2) {
      RQ::Row rows[2 * MT_GU_RP];
#pragma unroll
      for (int i = 0; i < 2 * MT_GU_RP; ++i) RQ::load_s(row_of(i), rows[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      refill(kq);
      for (int j = 0; j < n; ++j) {
        const uint32_t *pl = xpl + (size_t)(s_tok[base + j] * NCq + cl) * MT_CHW;
        RQ::XR xr;
        RQ::load_x(pl, reinterpret_cast<const float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB, xr);
        float v[2 * MT_GU_RP];
#pragma unroll
        for (int i = 0; i < 2 * MT_GU_RP; ++i) v[i] = RQ::dot_reg(rows[i], xr);
        emit(j, warp_sum_spread<2 * MT_GU_RP>(v));
      }
    } else {
      ScRow<2> rows[2 * MT_GU_RP];
#pragma unroll
      for (int i = 0; i < 2 * MT_GU_RP; ++i) load_scrow_s<2>(row_of(i), rows[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      refill(kq);
      for (int j = 0; j < n; ++j) {
        const uint32_t *pl = xpl + (size_t)(s_tok[base + j] * NCq + cl) * MT_CHW;
        RQ::XR xr;
        RQ::load_x(pl, reinterpret_cast<const float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB, xr);
        float v[2 * MT_GU_RP];
#pragma unroll
        for (int i = 0; i < 2 * MT_GU_RP; ++i) v[i] = scrow_dot<2>(rows[i], xr);
        emit(j, warp_sum_spread<2 * MT_GU_RP>(v));
      }
    }
  }
  // copies still in flight (only after a failed wait) land before the block ends
  if (producer)
    for (int qq = issued > MT_NS ? issued - MT_NS : 0; qq < issued; ++qq) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&S.full[qq % MT_NS], (qq / MT_NS) & 1))
        if (globaltimer_ns() - t0 > MT_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
    }
}

// ========================================================== h and planes ==

// h = SiLU(sum_q gp) * (sum_q up) for every routed pair in fixed-point planes
// (half a warp per 256-element block), and the shared activations as bf16
// hi + lo.
__global__ void __launch_bounds__(256) mt_h_kernel(const MtArgs a) {
  pdl_wait();     // gate/up partials complete and visible
  pdl_trigger();  // the down kernel may start streaming its weights
  const int lane = threadIdx.x & 31;
  const int NCf = a.F / MT_CHUNK, nbf = a.F / QK;
  const int64_t nblk = (int64_t)a.P * nbf;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u0 = gw; u0 < (nblk + 1) / 2; u0 += nw) {
    const int64_t bi = min(2 * u0 + (lane >> 4), nblk - 1);
    const int p = (int)(bi / nbf), b = (int)(bi % nbf);
    const int f0 = QK * b + 16 * (lane & 15);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
      for (int qq = 0; qq < a.KS; ++qq) {
        const float4 gq = __ldcg(reinterpret_cast<const float4 *>(a.gp + ((int64_t)qq * a.P + p) * a.F + f0 + j));
        const float4 uq = __ldcg(reinterpret_cast<const float4 *>(a.up + ((int64_t)qq * a.P + p) * a.F + f0 + j));
        g.x += gq.x; g.y += gq.y; g.z += gq.z; g.w += gq.w;
        u.x += uq.x; u.y += uq.y; u.z += uq.z; u.w += uq.w;
      }
      v[j] = silu(g.x) * u.x; v[j + 1] = silu(g.y) * u.y; v[j + 2] = silu(g.z) * u.z; v[j + 3] = silu(g.w) * u.w;
    }
    uint32_t *pl = a.hpl + ((int64_t)p * NCf + b / 4) * MT_CHW;
    RQ::digitize(v, b % 4, pl, reinterpret_cast<float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB);
  }
  const int64_t ns = (int64_t)a.T * a.Fs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns; i += (int64_t)gridDim.x * blockDim.x) {
    float g = 0.f, u = 0.f;
    for (int cc = 0; cc < a.D / MT_CHUNK; ++cc) {
      g += __ldcg(a.gs + (int64_t)cc * ns + i);
      u += __ldcg(a.us + (int64_t)cc * ns + i);
    }
    const float h = silu(g) * u;
    const __nv_bfloat16 hi = __float2bfloat16_rn(h);
    const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
    a.hs_hi[i] = __bfloat16_as_ushort(hi);
    a.hs_lo[i] = __bfloat16_as_ushort(lo);
  }
}

// =================================================================== down ==

struct DnLayout {
  size_t shared_off, planes_off, route_off, acc_off, total;
};

__host__ __device__ inline DnLayout dn_layout(int T, int NCqd, int E) {
  DnLayout L;
  L.shared_off = (size_t)MT_NS * MT_STAGE;
  L.planes_off = L.shared_off + al128(sizeof(MtShared));
  L.route_off = L.planes_off + al128((size_t)T * NCqd * MT_CHW * 4);
  L.acc_off = L.route_off + al128((size_t)3 * (E < MT_MAXP ? E : MT_MAXP) * 4);
  L.total = L.acc_off + (NCqd > 1 ? (size_t)MT_CONS * T * 8 * 4 : 0);
  return L;
}

__global__ void __launch_bounds__(MT_THREADS, 1)
    mt_dn_kernel(const MtArgs a, const __grid_constant__ CUtensorMap m_rdn, const __grid_constant__ CUtensorMap m_sd,
                 const __grid_constant__ CUtensorMap m_hh, const __grid_constant__ CUtensorMap m_hl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int T = a.T, P = a.P, D = a.D, Fs = a.Fs;
  const int G = gridDim.x, b = blockIdx.x;
  const int NCf = a.F / MT_CHUNK, NCqd = NCf / a.KSd, NCs = Fs / MT_CHUNK;
  const int q = b % a.KSd, bq = b / a.KSd;
  const int Gq = (G - q + a.KSd - 1) / a.KSd;
  const DnLayout L = dn_layout(T, NCqd, a.E);
  uint8_t *stages = smem;
  MtShared &S = *reinterpret_cast<MtShared *>(smem + L.shared_off);
  uint32_t *hpl = reinterpret_cast<uint32_t *>(smem + L.planes_off);
  const int maxu = a.E < MT_MAXP ? a.E : MT_MAXP;
  int32_t *s_used = reinterpret_cast<int32_t *>(smem + L.route_off);
  int32_t *s_base = s_used + maxu, *s_cnt = s_base + maxu;
  float *s_acc = reinterpret_cast<float *>(smem + L.acc_off);

  // shared-expert items: (128 rows of down, 1024-wide chunk of n_ff_shared),
  // dealt round-robin over all blocks; routed items: (expert slot, 64 rows),
  // the chunks of this block's slice each, contiguous per block
  const int S_items = Fs > 0 ? (D / MT_SH_ROWS) * NCs : 0;
  const int NB = MT_CHUNK / MT_BOX_K;
  const int n_sh = count_of(S_items, b, G);
  const int NG = D / MT_DN_NR;
  constexpr int C_SH = 24;  // a shared item's cost in the units of cost_boundary (12 tiles of bytes)

  // the route: written by the gate/up kernel, which completed before the h
  // kernel let this grid start
  const int nu = (int)__ldcg((const int *)(a.ctrl + C_NUSED));
  const bool bad_nu = nu < 0 || nu > maxu;
  for (int u = tid; u < (bad_nu ? 0 : nu); u += MT_THREADS) {
    int e = __ldcg(a.used + u);
    if (e < 0 || e >= a.E) { flag(a.status, ST_BAD_COUNT); e = 0; }
    const int b0 = __ldcg(a.offsets + e), n = __ldcg(a.offsets + e + 1) - b0;
    const bool ok = b0 >= 0 && n >= 0 && b0 + n <= P && n <= T;
    if (!ok) flag(a.status, ST_BAD_COUNT);
    s_used[u] = e;
    s_base[u] = ok ? b0 : 0;
    s_cnt[u] = ok ? n : 0;
  }
  if (tid == 0) {
    if (bad_nu) flag(a.status, ST_BAD_COUNT);
    for (int i = 0; i < MT_NS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], MT_CONS);
    }
    mbar_init(&S.planes_full, 1);
    mbar_init(&S.planes_empty, MT_CONS);
    S.abort_ = 0;
    S.nu = bad_nu ? 0 : nu;
    fence_mbar_init();
  }
  __syncthreads();
  const int nuu = S.nu;
  const int r0 = cost_boundary(bq, Gq, q, a.KSd, G, S_items, C_SH, nuu, s_cnt, NCqd, NG);
  const int r1 = cost_boundary(bq + 1, Gq, q, a.KSd, G, S_items, C_SH, nuu, s_cnt, NCqd, NG);
  const int n_rt = (r1 - r0) * NCqd;
  const int n_tiles = n_rt + n_sh * NB;

  // Lane 0 of the last warp issues the copies: routed down rows first (they
  // need no h, so the first stages stream while the h kernel still runs),
  // then the shared-expert tiles (weights and hs, after the h kernel).  The
  // planes of each expert's pairs are copied into shared memory when the
  // warps reach the expert's first tile, once all of them have released the
  // previous expert's planes.
  const bool producer = warp == MT_CONS - 1 && lane == 0;
  bool h_ready = false;  // (producer lane) the h kernel has completed
  // the tiles are issued in order: their coordinates advance without divisions
  int p_it = r0, p_cl = 0, p_u = r0 / NG, p_g = r0 % NG;         // routed: item it, chunk cl
  int p_kb = 0, p_cc = NCs > 0 ? b % NCs : 0, p_rs = NCs > 0 ? b / NCs : 0;  // shared: item b + G m, box kb
  const int p_gd = NCs > 0 ? G / NCs : 0, p_gm = NCs > 0 ? G % NCs : 0;
  auto issue = [&](int i) -> bool {
    const int st = i % MT_NS;
    if (i >= MT_NS && !mt_wait(&S.empty[st], ((i / MT_NS) & 1) ^ 1, S, a.status)) return false;
    uint8_t *dst = stages + (size_t)st * MT_STAGE;
    if (i < n_rt) {
      const int it = p_it, cl = p_cl, u = p_u, g = p_g;
      if (++p_cl == NCqd) {
        p_cl = 0;
        ++p_it;
        if (++p_g == NG) p_g = 0, ++p_u;
      }
      // an expert's first and last tiles: row group 0 or NG - 1, or the ends of this block's range
      const bool first = cl == 0 && (it == r0 || g == 0);
      const bool last = cl == NCqd - 1 && (it == r1 - 1 || g == NG - 1);
      S.desc[st] = make_int4(1, u, g, cl | (first ? 256 : 0) | (last ? 512 : 0));
      mbar_arrive_expect_tx(&S.full[st], (uint32_t)MT_DN_NR * MT_CB);
      tma3d(dst, &m_rdn, (q * NCqd + cl) * (MT_CB / 4), g * MT_DN_NR, s_used[u], &S.full[st]);
    } else {
      if (!h_ready) { pdl_wait(); h_ready = true; }  // hs is written by the h kernel
      const int kb = p_kb, cc = p_cc, rs = p_rs;
      if (++p_kb == NB) {
        p_kb = 0;
        p_cc += p_gm;
        p_rs += p_gd;
        if (p_cc >= NCs) p_cc -= NCs, ++p_rs;
      }
      S.desc[st] = make_int4(0, rs, kb, cc);
      mbar_arrive_expect_tx(&S.full[st], MT_SH_BOX + 2u * a.T8 * 128);
      const int kx = cc * MT_CHUNK + kb * MT_BOX_K;
      tma2d(dst, &m_sd, kx, rs * MT_SH_ROWS, &S.full[st]);
      tma2d(dst + MT_SH_BOX, &m_hh, kx, 0, &S.full[st]);
      tma2d(dst + MT_SH_BOX + a.T8 * 128, &m_hl, kx, 0, &S.full[st]);
    }
    return true;
  };
  int issued = 0;
  if (producer) {
    for (const CUtensorMap *m : {&m_rdn, &m_sd, &m_hh, &m_hl})
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
    while (issued < MT_NS && issued < n_tiles && issue(issued)) ++issued;
  }
  auto refill = [&](int kq) {
    if (producer && issued == kq + MT_NS && issued < n_tiles && issue(issued)) ++issued;
  };

  pdl_trigger();
  float c[MT_MAXT / 8][4];
#pragma unroll
  for (int tg = 0; tg < MT_MAXT / 8; ++tg) c[tg][0] = c[tg][1] = c[tg][2] = c[tg][3] = 0.f;
  const uint32_t stages_u32 = smem_u32(stages);
  int m_exp = 0;  // experts of this block so far
  for (int kq = 0; kq < n_tiles; ++kq) {
    const int st = kq % MT_NS;
    const bool got = mt_wait(&S.full[st], (kq / MT_NS) & 1, S, a.status);
    if (!got) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      continue;
    }
    const int4 d = S.desc[st];
    const uint32_t sbase = stages_u32 + (uint32_t)st * MT_STAGE;
    if (d.x == 0) {
      const int rs = d.y, kb = d.z, cc = d.w;
      shared_tile_mma(sbase, sbase + MT_SH_BOX, sbase + MT_SH_BOX + a.T8 * 128, true, a.T8, c, &S.empty[st]);
      refill(kq);
      if (kb == NB - 1) {
        store_shared_acc(c, a.ys + (int64_t)cc * T * D, D, rs * MT_SH_ROWS, T);
#pragma unroll
        for (int tg = 0; tg < MT_MAXT / 8; ++tg) c[tg][0] = c[tg][1] = c[tg][2] = c[tg][3] = 0.f;
      }
      continue;
    }
    const int u = d.y, g = d.z, cl = d.w & 255;
    const int base = s_base[u], n = s_cnt[u];
    const uint8_t *tile = stages + (size_t)st * MT_STAGE;
    constexpr int LV = 32 / MT_DN_R;  // lane LV i holds row i's value
    const int vi = lane / LV;
    const int drow = g * MT_DN_NR + warp * MT_DN_R + vi;
    auto emit = [&](int j, float tot) {
      if (lane % LV == 0) {
        if (NCqd > 1) {
          float *acc = s_acc + ((size_t)warp * T + j) * 8 + vi;
          tot = cl == 0 ? tot : *acc + tot;
          *acc = tot;
        }
        if (cl == NCqd - 1) a.y[((int64_t)q * P + base + j) * D + drow] = tot;
      }
    };
    // the first tile of an expert: its pair planes (copied here by the
    // producer lane, after every warp released the previous expert's)
    bool planes_ok = true;
    auto planes = [&]() {
      if (!(d.w & 256)) return;
      if (producer) {
        if (!h_ready) { pdl_wait(); h_ready = true; }
        bool ok = m_exp == 0 || mt_wait(&S.planes_empty, (m_exp - 1) & 1, S, a.status);
        if (ok) {
          const uint32_t pb = (uint32_t)(NCqd * MT_CHW * 4);
          mbar_arrive_expect_tx(&S.planes_full, pb * (uint32_t)n);
          for (int j = 0; j < n; ++j)
            bulk_g2s(hpl + (size_t)j * NCqd * MT_CHW, a.hpl + ((int64_t)(base + j) * NCf + q * NCqd) * MT_CHW, pb,
                     &S.planes_full);
        }
      }
      planes_ok = mt_wait(&S.planes_full, m_exp & 1, S, a.status);
      ++m_exp;
    };
    if (n <= 2) {
      RQ::Row rr[MT_DN_R];
#pragma unroll
      for (int i = 0; i < MT_DN_R; ++i) RQ::load_s(tile + (size_t)(warp * MT_DN_R + i) * MT_CB, rr[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      refill(kq);
      planes();
      for (int j = 0; planes_ok && j < n; ++j) {
        const uint32_t *pl = hpl + (size_t)(j * NCqd + cl) * MT_CHW;
        RQ::XR xr;
        RQ::load_x(pl, reinterpret_cast<const float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB, xr);
        float v[MT_DN_R];
#pragma unroll
        for (int i = 0; i < MT_DN_R; ++i) v[i] = RQ::dot_reg(rr[i], xr);
        emit(j, warp_sum_spread<MT_DN_R>(v));
      }
    } else {
      ScRow<2> rr[MT_DN_R];
#pragma unroll
      for (int i = 0; i < MT_DN_R; ++i) load_scrow_s<2>(tile + (size_t)(warp * MT_DN_R + i) * MT_CB, rr[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[st]);
      refill(kq);
      planes();
      for (int j = 0; planes_ok && j < n; ++j) {
        const uint32_t *pl = hpl + (size_t)(j * NCqd + cl) * MT_CHW;
        RQ::XR xr;
        RQ::load_x(pl, reinterpret_cast<const float *>(pl + RQ::NPL * (MT_CHUNK / RQ::SUB)), MT_CHUNK / RQ::SUB, xr);
        float v[MT_DN_R];
#pragma unroll
        for (int i = 0; i < MT_DN_R; ++i) v[i] = scrow_dot<2>(rr[i], xr);
        emit(j, warp_sum_spread<MT_DN_R>(v));
      }
    }
    if (d.w & 512) {  // the expert's last tile: its planes may be replaced
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.planes_empty);
    }
  }
  if (producer) {
    // copies still in flight (only after a failed wait) land before the block ends
    for (int qq = issued > MT_NS ? issued - MT_NS : 0; qq < issued; ++qq) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&S.full[qq % MT_NS], (qq / MT_NS) & 1))
        if (globaltimer_ns() - t0 > MT_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
    }
    if (m_exp > 0) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&S.planes_full, (m_exp - 1) & 1))
        if (globaltimer_ns() - t0 > MT_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
    }
    // this grid completes only after the h kernel (whose inputs the next
    // layer's gate/up kernel overwrites) has
    if (!h_ready) pdl_wait();
  }
}

// ================================================================ combine ==

// out[t] (+)= sum_c ys[c][t] + sum_j w[t][j] * (sum_q y[q][pos[t][j]]), slot
// order j, partial sums in order.
__global__ void __launch_bounds__(256) mt_combine_kernel(const MtArgs a) {
  pdl_wait();
  const int d4 = a.D / 4;
  const int64_t n = (int64_t)a.T * d4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / d4;
    const int c = (int)(i % d4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int qq = 0; qq < a.Fs / MT_CHUNK; ++qq) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.ys + ((int64_t)qq * a.T + t) * a.D) + c);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    for (int j = 0; j < a.k; ++j) {
      const int pj = __ldcg(a.pos + t * a.k + j);
      const float wj = __ldcg(a.w + t * a.k + j);
      float4 yv = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int qq = 0; qq < a.KSd; ++qq) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.y + ((int64_t)qq * a.P + pj) * a.D) + c);
        yv.x += v.x; yv.y += v.y; yv.z += v.z; yv.w += v.w;
      }
      acc.x = fmaf(wj, yv.x, acc.x); acc.y = fmaf(wj, yv.y, acc.y);
      acc.z = fmaf(wj, yv.z, acc.z); acc.w = fmaf(wj, yv.w, acc.w);
    }
    float4 *o = reinterpret_cast<float4 *>(a.out + t * a.D) + c;
    if (a.accumulate) {
      const float4 r = *o;
      acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
    }
    *o = acc;
  }
}

// ------------------------------------------------------------- host side --

// Slices: the smallest power of two dividing n_chunks with tokens x
// chunks-per-slice within what a block holds.
int slices_for(int n_chunks, int T) {
  for (int s = 1; s <= n_chunks; s <<= 1)
    if (n_chunks % s == 0 && (int64_t)T * (n_chunks / s) <= MT_TCH) return s;
  return 0;
}

template <typename K>
cudaError_t launch_pdl_mt(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          const MtArgs &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename K, typename... M>
cudaError_t launch_pdl_maps(K kern, dim3 grid, size_t smem, cudaStream_t s, const MtArgs &a, const M &...maps) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(MT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, maps...);
}

// Kernel attributes, set once per device.
cudaError_t mt_setup() {
  static OncePerDevice once;
  return once_per_device(once, []() {
    const int lim = (int)MT_SMEM_LIMIT;
    cudaError_t e = cudaFuncSetAttribute(mt_gu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(mt_dn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    return e;
  });
}

size_t gu_smem(const Shape &sh, int64_t T) {
  const int KS = slices_for(sh.D / MT_CHUNK, (int)T);
  return 1024 + gu_layout((int)T, sh.D / MT_CHUNK / std::max(KS, 1), sh.E, (int)(T * sh.k)).total;
}

size_t dn_smem(const Shape &sh, int64_t T) {
  const int KSd = slices_for(sh.F / MT_CHUNK, (int)T);
  return 1024 + dn_layout((int)T, sh.F / MT_CHUNK / std::max(KSd, 1), sh.E).total;
}

}  // namespace

bool decode_mt_supported(const Shape &sh, int64_t T) {
  if (sh.fmt != DS_Q2_K) return false;
  if (T < MT_MIN_T || T > MT_MAX_T || T * sh.k > MT_MAXP) return false;
  if (sh.x_dtype != DS_BF16 || sh.router_dtype != DS_BF16) return false;
  if (sh.D % MT_CHUNK || sh.F % MT_CHUNK || sh.Fs % MT_CHUNK) return false;
  if (sh.D > 8192 || sh.F > 8192 || sh.E > 1024 || sh.k > 16) return false;
  if (slices_for(sh.D / MT_CHUNK, (int)T) == 0 || slices_for(sh.F / MT_CHUNK, (int)T) == 0) return false;
  if (gu_smem(sh, T) > MT_SMEM_LIMIT || dn_smem(sh, T) > MT_SMEM_LIMIT) return false;
  return encode_fn() != nullptr;
}

size_t decode_mt_workspace(const Shape &sh, int64_t T) {
  const int64_t P = T * sh.k;
  const int KS = std::max(slices_for(sh.D / MT_CHUNK, (int)T), 1);
  const int KSd = std::max(slices_for(sh.F / MT_CHUNK, (int)T), 1);
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t fs = (size_t)std::max(sh.Fs, 1);
  const size_t NCd = sh.D / MT_CHUNK, NCs = std::max(sh.Fs / MT_CHUNK, 1);
  return 2 * up(4 * (size_t)KS * P * sh.F) + 2 * up(4 * NCd * T * fs) +
         up(4 * (size_t)P * (sh.F / MT_CHUNK) * MT_CHW) + 2 * up(2 * (size_t)T * fs) +
         up(4 * (size_t)KSd * P * sh.D) + up(4 * NCs * T * sh.D);
}

cudaError_t launch_decode_mt(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk, float *out,
                             bool accumulate, void *mt_ws, cudaStream_t s) {
  cudaError_t e = mt_setup();
  if (e != cudaSuccess) return e;
  const int G = device_sms();
  if (!G) return cudaErrorNoDevice;
  const int T = (int)wk.T, P = T * sh.k;
  const int KS = slices_for(sh.D / MT_CHUNK, T), KSd = slices_for(sh.F / MT_CHUNK, T);
  if (KS == 0 || KSd == 0) return cudaErrorInvalidValue;
  MtArgs a{};
  a.D = sh.D; a.E = sh.E; a.F = sh.F; a.Fs = sh.Fs; a.k = sh.k; a.T = T; a.T8 = (T + 7) & ~7; a.P = P;
  a.KS = KS; a.KSd = KSd;
  a.routed_scale = sh.routed_scale;
  a.logit_scale = sh.logit_scale;
  a.unbias = sh.bias_select_only ? W.router_bias : nullptr;
  a.experts = W.experts;
  a.expert_bytes = sh.expert_bytes();
  a.gate_bytes = sh.gate_bytes();
  a.x = (const uint16_t *)x;
  a.logits = wk.logits;
  a.ids = wk.ids; a.w = wk.w; a.counts = wk.counts; a.offsets = wk.offsets; a.perm = wk.perm; a.pos = wk.pos;
  a.used = wk.used;
  a.ctrl = wk.ctrl;
  // workspace carve-up (see decode_mt_workspace)
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t fs = (size_t)std::max(sh.Fs, 1);
  char *p = static_cast<char *>(mt_ws);
  a.gp = reinterpret_cast<float *>(p); p += up(4 * (size_t)KS * P * sh.F);
  a.up = reinterpret_cast<float *>(p); p += up(4 * (size_t)KS * P * sh.F);
  const size_t NCd = sh.D / MT_CHUNK;
  a.gs = reinterpret_cast<float *>(p); p += up(4 * NCd * T * fs);
  a.us = reinterpret_cast<float *>(p); p += up(4 * NCd * T * fs);
  a.hpl = reinterpret_cast<uint32_t *>(p); p += up(4 * (size_t)P * (sh.F / MT_CHUNK) * MT_CHW);
  a.hs_hi = reinterpret_cast<uint16_t *>(p); p += up(2 * (size_t)T * fs);
  a.hs_lo = reinterpret_cast<uint16_t *>(p); p += up(2 * (size_t)T * fs);
  a.y = reinterpret_cast<float *>(p); p += up(4 * (size_t)KSd * P * sh.D);
  a.ys = reinterpret_cast<float *>(p);
  a.out = out;
  a.accumulate = accumulate ? 1 : 0;
  a.status = status_word();

  // tensor maps: routed rows as 32-bit words; shared rows, x and hs as bf16
  // tiles in the 128-byte swizzle
  CUtensorMap m_rgu, m_rdn, m_sg, m_su, m_sd, m_x, m_hh, m_hl;
  const void *sgb = sh.Fs > 0 ? (const void *)W.shared_gate : (const void *)W.experts;
  const void *sub = sh.Fs > 0 ? (const void *)W.shared_up : (const void *)W.experts;
  const void *sdb = sh.Fs > 0 ? (const void *)W.shared_down : (const void *)W.experts;
  const int64_t fsr = sh.Fs > 0 ? sh.Fs : MT_SH_ROWS;
  if (!make_words_map(&m_rgu, W.experts, (int64_t)(sh.D / QK) * QB, 2 * (int64_t)sh.F, sh.E, sh.expert_bytes(),
                      MT_CB / 4, MT_GU_NR) ||
      !make_words_map(&m_rdn, W.experts + 2 * sh.gate_bytes(), (int64_t)(sh.F / QK) * QB, sh.D, sh.E,
                      sh.expert_bytes(), MT_CB / 4, MT_DN_NR) ||
      !make_map(&m_sg, sgb, fsr, sh.D, MT_SH_ROWS, true) || !make_map(&m_su, sub, fsr, sh.D, MT_SH_ROWS, true) ||
      !make_map(&m_sd, sdb, sh.D, sh.Fs > 0 ? sh.Fs : MT_BOX_K, MT_SH_ROWS, true) ||
      !make_map(&m_x, x, T, sh.D, a.T8, true) ||
      !make_map(&m_hh, a.hs_hi, T, sh.Fs > 0 ? sh.Fs : MT_BOX_K, a.T8, true) ||
      !make_map(&m_hl, a.hs_lo, T, sh.Fs > 0 ? sh.Fs : MT_BOX_K, a.T8, true))
    return cudaErrorInvalidValue;

  if ((e = launch_pdl_maps(mt_gu_kernel, dim3(G), gu_smem(sh, T), s, a, m_rgu, m_sg, m_su, m_x)) != cudaSuccess)
    return e;
  if ((e = launch_pdl_mt(mt_h_kernel, dim3(G), dim3(256), 0, s, true, a)) != cudaSuccess) return e;
  if ((e = launch_pdl_maps(mt_dn_kernel, dim3(G), dn_smem(sh, T), s, a, m_rdn, m_sd, m_hh, m_hl)) != cudaSuccess)
    return e;
  return launch_pdl_mt(mt_combine_kernel, dim3(G), dim3(256), 0, s, true, a);
}

}  // namespace dsm
