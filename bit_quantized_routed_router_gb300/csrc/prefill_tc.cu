// Large-batch (prefill) expert FFNs on the 5th-generation tensor cores.
//
// What it computes is the expert part of the layer of "Understanding Dwarf
// Star" 5.3.2 / 5.3.4 / 5.3.7: for every routed expert e and its tokens,
// h = SiLU(X_e Wg_e^T) * (X_e Wu_e^T) and y = h Wd_e^T with the Q2_K weights
// of 3.3.3 dequantised on the fly (2.8.1-2.8.2), plus the always-active bf16
// shared expert over all tokens.  The router, selection, route and the
// combine out = y_shared + sum_j w_j y_j run in their own kernels.
//
// Both contractions run "weights as M": a tile is 128 weight rows (the f
// rows of gate and up, or the d rows of down) times up to N tokens of one
// expert (N rounded up to a multiple of 16; at most 128, or 256 when the
// tile plan picks the wide layout for a launch), so an expert with 96
// tokens wastes no more than 15 columns.  Per tile and 64-wide K step:
//
//   dequant warps  Q2_K rows -> fp16 in the 128-byte swizzled K-major layout
//                  of the MMA, from raw copies (96 bytes per row holding one
//                  84-byte block, 128 rows per tensor copy) that the copy
//                  warp stages in shared memory ahead of them;
//   copy warp      bulk-tensor (TMA) loads of the token rows (fp16) and, for
//                  the dense shared expert, of its weight rows;
//   MMA thread     tcgen05.mma kind::f16, fp32 accumulators in tensor memory
//                  (two accumulator buffers, so the epilogue of one tile
//                  overlaps the main loop of the next; a tile wider than 128
//                  tokens takes both);
//   epilogue warps tcgen05.ld of the accumulators: SiLU(g) * u -> h (fp16),
//                  or y (fp32).
//
// Dequantised weights are exact fp32 values d*sc*q - dmin*m rounded once to
// fp16.  Within every group of 16 consecutive K indices the operands are
// stored in a fixed order (position p holds index 4 (p mod 4) + p / 4) that
// makes the dequantisation a byte permutation; the activations are written
// in the same order, and a K-sum does not depend on the order of its terms.
#include <cuda.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dsm {
namespace {

constexpr int TC_BM = 128;                 // weight rows per tile (MMA M)
constexpr int TC_BK = 64;                  // K per stage: one 128-byte swizzle row
constexpr int TC_NGU = 128;                // tokens per gate/up or down tile at most, Q4_K
constexpr int TC_NDN = 128;                //   (and the chunk the workspace is sized for)
constexpr int TC_NWIDE = 256;              // tokens per gate/up or down tile at most, Q2_K
constexpr int TC_NRT = 256;                // tokens per router tile at most
constexpr uint32_t TC_TILE_BYTES = TC_BM * 128;       // one 128 x 64 operand tile (16 KB)
constexpr uint32_t TC_RAW_ROW = 96;        // bytes copied per weight row and 256-weight block (Q2_K)
constexpr uint32_t TC_RAW_ROW_Q4 = Q4B;    // Q4_K: the 144-byte block itself (16-byte aligned)
constexpr int TC_MAX_STAGES = 5, TC_MAX_RAW = 3;
constexpr int TC_TILE_CACHE = 128;         // a block's first tiles, copied to shared memory
constexpr int TC_EPI = 4, TC_DQ = 8;       // epilogue and dequant warps
constexpr int TC_MMA_WARP = TC_EPI, TC_TMA_WARP = TC_EPI + 1, TC_DQ0 = TC_EPI + 2;
constexpr int TC_THREADS = (TC_EPI + 2 + TC_DQ) * 32;
constexpr uint64_t TC_LIMIT_NS = 2000000000ull;
constexpr uint32_t TC_TMEM_COLS = 512;

// Tile of a contraction: kind 0 = routed expert e, 1 = shared expert; brow =
// first row of the token operand (a route position for routed tiles, a token
// for shared ones); n tokens; blk = 128-row block of weights.
struct TcTile {
  int kind, e, brow, n, blk;
};

// The three contractions of the path.
enum { MODE_GU = 0, MODE_DN = 1, MODE_ROUTER = 2 };

// Pipeline shape per contraction: a stage holds A_TILES weight tiles (gate
// and up, or one) and a token tile of NMAX rows; RAW slots of raw blocks
// (one per 256-wide K block) feed the dequant warps.  A Q2_K raw slot is
// free again as soon as the dequant warps hold its rows in registers, so one
// slot keeps a block in flight, and the ring has one of two layouts, which
// the tile plan chooses per launch: four stages of up to 128 tokens, or
// (when experts with more than 128 tokens make it worth it) three stages of
// up to 256 tokens, so that such an expert is dequantised once per 256 of
// its tokens instead of per 128.  Q4_K blocks (144 bytes) are read from the
// slot stage by stage, so Q4_K keeps two raw slots and three stages of 128
// tokens within the shared memory of a block.
template <int MODE, int FMT = DS_Q2_K>
struct TcCfg {
  static constexpr int A_TILES = MODE == MODE_ROUTER ? 1 : 2;  // gate + up, or two 128-row down blocks
  static constexpr int NMAX = MODE == MODE_ROUTER ? TC_NRT : TC_NGU;
  static constexpr int STAGES = MODE == MODE_ROUTER ? 4 : FMT == DS_Q4_K ? 3 : 4;
  static constexpr int RAW = MODE == MODE_ROUTER ? 1 : FMT == DS_Q4_K ? 2 : 1;
  static constexpr uint32_t RAW_ROW = FMT == DS_Q4_K ? TC_RAW_ROW_Q4 : TC_RAW_ROW;
  static constexpr uint32_t STAGE_BYTES = (A_TILES + NMAX / 128) * TC_TILE_BYTES;
  static constexpr uint32_t RAW_BYTES = A_TILES * TC_BM * RAW_ROW;
  // the wide layout
  static constexpr bool WIDE = MODE != MODE_ROUTER && FMT == DS_Q2_K;
  static constexpr int NMAX_W = TC_NWIDE, STAGES_W = 3;
  static constexpr uint32_t STAGE_BYTES_W = (A_TILES + NMAX_W / 128) * TC_TILE_BYTES;
  static constexpr uint32_t RING_BYTES =
      WIDE && STAGES_W * STAGE_BYTES_W > STAGES * STAGE_BYTES ? STAGES_W * STAGE_BYTES_W : STAGES * STAGE_BYTES;
};

struct TcArgs {
  int D, F, Fs, P, T, E;
  int router_tiles;        // MODE_ROUTER: tiles (E / 128 rounded up) x (T / 256 rounded up)
  float *logits;           // MODE_ROUTER: [T][E]
  const float *bias;       // MODE_ROUTER: [E] or null
  const uint8_t *experts;
  int64_t expert_bytes, gate_bytes;
  const int4 *tiles;
  const int *n_tiles;
  const int *wide;         // non-zero: the plan chose the wide layout (Q2_K gate/up and down)
  uint16_t *h16;  // fp16: routed rows [P][F] (K order permuted), then shared rows [T][Fs]
  float *y;       // [P][D] routed outputs, perm order
  float *ys;      // [T][D] shared output
  unsigned *status;
};

__device__ __forceinline__ TcTile tile_at(const int4 *list, int i) {
  const int4 v = list[i];
  return TcTile{v.x, v.y, v.z, v.w & 0xFFFF, v.w >> 16};
}

// ------------------------------------------------------------ PTX wrappers --

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row groups 1024 bytes apart), start address `addr`.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset: 8 rows x 128 bytes
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands
// K-major, M = 128, N = n (a multiple of 16 up to 256); bf16 when ab_bf16.
__device__ __forceinline__ uint32_t f16_idesc(int n, bool ab_bf16) {
  uint32_t d = 1u << 4;                   // D format fp32
  if (ab_bf16) d |= (1u << 7) | (1u << 10);
  d |= (uint32_t)(n >> 3) << 17;
  d |= (uint32_t)(TC_BM >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcShared {
  uint64_t full[TC_MAX_STAGES], empty[TC_MAX_STAGES];
  uint64_t raw_full[TC_MAX_RAW], raw_empty[TC_MAX_RAW];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem;
  int abort_;
  int4 tiles[TC_TILE_CACHE];
};

// Bounded wait for the phase of `bar` with parity `par`.  Each try lets the
// thread sleep until the phase completes (or 20 us pass), so waiting warps
// do not take issue slots from the dequantising ones.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t par, TcShared &S, unsigned *status) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, par, 20000u)) {
    if (*(volatile int *)&S.abort_) return false;
    if (globaltimer_ns() - t0 > TC_LIMIT_NS) {
      flag(status, ST_TIMEOUT);
      *(volatile int *)&S.abort_ = 1;
      return false;
    }
  }
  return true;
}

// K of a tile.
template <int MODE>
__device__ __forceinline__ int tile_k(const TcArgs &a, const TcTile &t) {
  return MODE == MODE_DN ? (t.kind == 0 ? a.F : a.Fs) : a.D;
}

// Tile i of this launch: from the list, or (router) by position.
template <int MODE>
__device__ __forceinline__ TcTile get_tile(const TcArgs &a, int i) {
  if (MODE == MODE_ROUTER) {
    const int neb = (a.E + TC_BM - 1) / TC_BM;
    const int t0 = (i / neb) * TC_NRT;
    return TcTile{1, 0, t0, min(TC_NRT, a.T - t0), i % neb};
  }
  return tile_at(a.tiles, i);
}

// The fp16 pair (v[qa], v[qb]) for the selector nibbles built below: lut_lo
// holds v0 | v1 << 16, lut_hi v2 | v3 << 16.
__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
  return r;
}

// Dequantise one sub-block (16 weights) of a Q2_K block from its code word
// and scale byte (sc low nibble, m high nibble), d and dmin, into the two
// 16-byte chunks of its K positions (the order described at the top of the
// file): chunk 0 = positions 0-7, chunk 1 = positions 8-15.  The four values
// v_q = fp16(d sc q - dmin m) are computed exactly in fp32 and rounded once;
// each weight is then a byte permutation of them, selected by its code.
__device__ __forceinline__ void dequant_codes(uint32_t codes, uint32_t scm, float d, float dmin, uint4 &c0,
                                              uint4 &c1) {
  const float av = d * (float)(scm & 15u), bv = dmin * (float)(scm >> 4);  // both exact
  const __half2 v01 = __floats2half2_rn(-bv, fmaf(av, 1.f, -bv));
  const __half2 v23 = __floats2half2_rn(fmaf(av, 2.f, -bv), fmaf(av, 3.f, -bv));
  const uint32_t lo = *reinterpret_cast<const uint32_t *>(&v01);
  const uint32_t hi = *reinterpret_cast<const uint32_t *>(&v23);
  uint32_t w[8];
#pragma unroll
  for (int sh = 0; sh < 4; ++sh) {
    const uint32_t y = (codes >> (2 * sh)) & 0x03030303u;
    const uint32_t sel = y * 0x22u + 0x10101010u;
    w[2 * sh] = prmt(lo, hi, sel);
    w[2 * sh + 1] = prmt(lo, hi, sel >> 16);
  }
  c0 = make_uint4(w[0], w[1], w[2], w[3]);
  c1 = make_uint4(w[4], w[5], w[6], w[7]);
}

// One Q4_K sub-block (32 weights: code words cw[0..3], weight 8 c + 2 b in
// the low nibble of byte b of word c, 8 c + 2 b + 1 in the high nibble) as
// two 16-groups of fp16 in the permuted K order (position p of a group holds
// index 4 (p mod 4) + p / 4): four 16-byte chunks.  Each weight is the exact
// fp32 value q * (d sc) - dmin m (one rounding: both products are exact)
// rounded to fp16; q becomes a float through the exponent of 2^23 (exact).
// Sixteen levels do not fit the Q2_K byte permutation, which selects among
// four fp16 values.
__device__ __forceinline__ float q4_code_f(uint32_t cw, int shift) {
  return __uint_as_float(((cw >> shift) & 0xFu) | 0x4B000000u) - 8388608.0f;
}

__device__ __forceinline__ void dequant_q4_sub(const uint4 codes, float dsc, float dmm, uint4 out[4]) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // 16-group: weights 16 h .. 16 h + 15
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // positions 2 i, 2 i + 1
      float v[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int pp = 2 * i + t, k = 4 * (pp & 3) + (pp >> 2);  // index within the group
        const int w = 16 * h + k;                                   // weight within the sub-block
        v[t] = fmaf(q4_code_f(cw[w >> 3], 8 * ((w & 7) >> 1) + 4 * (w & 1)), dsc, -dmm);
      }
      const __half2 hv = __floats2half2_rn(v[0], v[1]);
      o[i] = *reinterpret_cast<const uint32_t *>(&hv);
    }
    out[2 * h] = make_uint4(o[0], o[1], o[2], o[3]);
    out[2 * h + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Operand tiles are 128 rows x 64 K-elements in the 128-byte swizzle of the
// MMA descriptors: 16-byte chunk c (K elements 8c..8c+7) of row r sits at
// byte r * 128 + ((c ^ (r mod 8)) * 16) of the 1024-byte aligned tile.

template <int MODE, int FMT = DS_Q2_K>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tm_raw,
                   const __grid_constant__ CUtensorMap tm_b_r32, const __grid_constant__ CUtensorMap tm_b_r64,
                   const __grid_constant__ CUtensorMap tm_b_r96, const __grid_constant__ CUtensorMap tm_b_r128,
                   const __grid_constant__ CUtensorMap tm_b_routed, const __grid_constant__ CUtensorMap tm_b_shared,
                   const __grid_constant__ CUtensorMap tm_b_shared_w, const __grid_constant__ CUtensorMap tm_a0,
                   const __grid_constant__ CUtensorMap tm_a1) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the swizzle pattern repeats every 1024 bytes);
  // derived from the array itself so that accesses stay shared-memory ones
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;
  using C = TcCfg<MODE, FMT>;
  constexpr int TC_RAW_SLOTS = C::RAW;
  constexpr uint32_t TC_RAW_BYTES = C::RAW_BYTES;
  // the ring layout of this launch (every role reads the same word)
  const bool wl = C::WIDE && *a.wide != 0;
  const int TC_STAGES = wl ? C::STAGES_W : C::STAGES, NMAX = wl ? C::NMAX_W : C::NMAX;
  const uint32_t TC_STAGE_BYTES = wl ? C::STAGE_BYTES_W : C::STAGE_BYTES;
  uint8_t *raw = smem + C::RING_BYTES;
  TcShared &S = *reinterpret_cast<TcShared *>(raw + TC_RAW_SLOTS * TC_RAW_BYTES);
  constexpr bool GU = MODE == MODE_GU;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  const int n_tiles = MODE == MODE_ROUTER ? a.router_tiles : *a.n_tiles;

  if (MODE != MODE_ROUTER)
    for (int j = threadIdx.x; j < TC_TILE_CACHE && bid + G * j < n_tiles; j += TC_THREADS) S.tiles[j] = a.tiles[bid + G * j];
  // tile i of this block
  auto tile_of = [&](int i) -> TcTile {
    if (MODE == MODE_ROUTER) return get_tile<MODE>(a, bid + G * i);
    const int4 v = i < TC_TILE_CACHE ? S.tiles[i] : a.tiles[bid + G * i];
    return TcTile{v.x, v.y, v.z, v.w & 0xFFFF, v.w >> 16};
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < TC_STAGES; ++i) {
      mbar_init(&S.full[i], 1 + TC_DQ);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < TC_RAW_SLOTS; ++i) {
      mbar_init(&S.raw_full[i], 1);
      mbar_init(&S.raw_empty[i], TC_DQ);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], TC_EPI);
    }
    mbar_init(&S.drain, 1);
    S.abort_ = 0;
    fence_mbar_init();
  }
  if (warp == TC_MMA_WARP) {  // the whole warp allocates the accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&S.tmem)),
                 "r"(TC_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;

  if (warp == TC_TMA_WARP) {
    // -------------------------------------------------- copies (one warp) --
    // Raw blocks (one copy per weight row and 256-wide K block: a 96-byte
    // window holding the Q2_K block, or the 144-byte Q4_K block) of the
    // routed tiles run ahead of the stages: when the stages of the routed
    // block c begin, blocks up to c + RAW - 1 are issued (waiting for their
    // slots), and block c + RAW as soon as its slot is free (checked before
    // every stage, never waited for).  (ri, rkb) walks the routed blocks in
    // the order the dequant warps consume them.
    if (lane == 0) {  // descriptors into the TMA unit's cache before the first copies
      const CUtensorMap *maps[10] = {&tm_raw,      &tm_b_r32,    &tm_b_r64,      &tm_b_r96, &tm_b_r128,
                                     &tm_b_routed, &tm_b_shared, &tm_b_shared_w, &tm_a0,    &tm_a1};
      for (int m = 0; m < 10; ++m)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(maps[m])) : "memory");
    }
    int st_it = 0, rawq = 0, rawpos = 0, ri = 0, rkb = 0;
    int sl = 0, ph = 0;  // slot and phase of stage st_it (no division by the runtime stage count)
    bool ok = true;
    auto issue_raw = [&](bool wait) -> int {  // 1 issued, 0 none left (or slot busy), -1 failed wait
      for (;;) {
        if (bid + G * ri >= n_tiles) return 0;
        const TcTile t = tile_of(ri);
        if (t.kind == 0 && rkb < tile_k<MODE>(a, t) / QK) break;
        ++ri;
        rkb = 0;
      }
      const TcTile t = tile_of(ri);
      const int slot = rawq % TC_RAW_SLOTS;
      if (rawq >= TC_RAW_SLOTS) {
        int w = 1;
        if (!wait) {
          if (lane == 0) w = mbar_test_wait(&S.raw_empty[slot], ((rawq / TC_RAW_SLOTS) & 1) ^ 1);
          if (!__shfl_sync(0xffffffffu, w, 0)) return 0;
        } else {
          if (lane == 0) w = tc_wait(&S.raw_empty[slot], ((rawq / TC_RAW_SLOTS) & 1) ^ 1, S, a.status);
          if (!__shfl_sync(0xffffffffu, w, 0)) return -1;
        }
      }
      const int rows = 2 * TC_BM;
      if (lane == 0) {
        // words [x, x + 24) of 128 weight rows: the 96-byte window, 16-byte
        // aligned, that holds block rkb of each row
        mbar_arrive_expect_tx(&S.raw_full[slot], rows * C::RAW_ROW);
        const int xw = FMT == DS_Q4_K ? (int)((uint32_t)(Q4B * rkb) >> 2) : (int)(((uint32_t)(QB * rkb) & ~15u) >> 2);
        uint8_t *dst = raw + (size_t)slot * TC_RAW_BYTES;
        // gate/up: rows blk*128 of gate and of up; down: rows blk*256 and blk*256 + 128
        const int y0 = GU ? t.blk * TC_BM : 2 * t.blk * TC_BM;
        tma_load_3d(dst, &tm_raw, xw, y0, t.e, &S.raw_full[slot]);
        tma_load_3d(dst + TC_BM * C::RAW_ROW, &tm_raw, xw, GU ? a.F + y0 : y0 + TC_BM, t.e, &S.raw_full[slot]);
      }
      __syncwarp();
      ++rawq;
      ++rkb;
      return 1;
    };
    for (int i = 0; ok && bid + G * i < n_tiles; ++i) {
      const TcTile t = tile_of(i);
      const int nk = tile_k<MODE>(a, t) / TC_BK;
      const bool routed = t.kind == 0;
      for (int kc = 0; ok && kc < nk; ++kc) {
        if (routed && (kc & 3) == 0) {
          ++rawpos;
          while (rawq < rawpos + TC_RAW_SLOTS - 1) {
            const int r = issue_raw(true);
            if (r < 0) ok = false;
            if (r <= 0) break;
          }
          if (!ok) break;
        }
        if (rawq < rawpos + TC_RAW_SLOTS) issue_raw(false);  // one block further once its slot is free
        const int s = sl;
        if (st_it >= TC_STAGES) {
          int w = 1;
          if (lane == 0) w = tc_wait(&S.empty[s], ph ^ 1, S, a.status);
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        uint8_t *stage = stages + (size_t)s * TC_STAGE_BYTES;
        if (lane == 0) {
          // one box of token rows: a routed tile's width rounded up to 32
          // (up to 128 tokens) or NMAX (wider routed tiles, and shared ones);
          // rows past the tile's tokens only feed accumulator columns that
          // are never read
          const int bsel = routed && MODE != MODE_ROUTER ? (t.n > 128 ? 4 : (t.n - 1) >> 5) : 4;
          const CUtensorMap *bm = !routed       ? (wl ? &tm_b_shared_w : &tm_b_shared)
                                  : bsel == 0 ? &tm_b_r32
                                  : bsel == 1 ? &tm_b_r64
                                  : bsel == 2 ? &tm_b_r96
                                  : bsel == 3 ? &tm_b_r128
                                              : &tm_b_routed;
          uint32_t bytes = (uint32_t)(bsel < 4 ? 32 * (bsel + 1) : NMAX) * 128;
          if (!routed) bytes += C::A_TILES * TC_TILE_BYTES;
          mbar_arrive_expect_tx(&S.full[s], bytes);
          uint8_t *bdst = stage + C::A_TILES * TC_TILE_BYTES;
          tma_load_2d(bdst, bm, kc * TC_BK, t.brow, &S.full[s]);
          if (!routed) {
            if (GU) {
              tma_load_2d(stage, &tm_a0, kc * TC_BK, t.blk * TC_BM, &S.full[s]);
              tma_load_2d(stage + TC_TILE_BYTES, &tm_a1, kc * TC_BK, t.blk * TC_BM, &S.full[s]);
            } else if (MODE == MODE_DN) {
              tma_load_2d(stage, &tm_a0, kc * TC_BK, 2 * t.blk * TC_BM, &S.full[s]);
              tma_load_2d(stage + TC_TILE_BYTES, &tm_a0, kc * TC_BK, 2 * t.blk * TC_BM + TC_BM, &S.full[s]);
            } else {
              tma_load_2d(stage, &tm_a0, kc * TC_BK, t.blk * TC_BM, &S.full[s]);
            }
          }
        }
        __syncwarp();
        ++st_it;
        if (++sl == TC_STAGES) sl = 0, ph ^= 1;
      }
    }
    // every copy issued has landed before the block may end
    if (lane == 0) {
      for (int q = st_it > TC_STAGES ? st_it - TC_STAGES : 0; q < st_it; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&S.full[q % TC_STAGES], (q / TC_STAGES) & 1))
          if (globaltimer_ns() - t0 > TC_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
      }
      for (int q = rawq > TC_RAW_SLOTS ? rawq - TC_RAW_SLOTS : 0; q < rawq; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&S.raw_full[q % TC_RAW_SLOTS], (q / TC_RAW_SLOTS) & 1))
          if (globaltimer_ns() - t0 > TC_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
      }
    }
  } else if (warp >= TC_DQ0) {
    // ------------------------------------------------------ dequant warps --
    // Thread dt owns one weight row of every stage, all four of its
    // sub-blocks: gate/up: row dt (gate rows 0-127, then up rows); down: row
    // dt of the two 128-row blocks.  Its raw and destination offsets are fixed.
    const int dt = threadIdx.x - TC_DQ0 * 32;  // 0 .. 255
    const int r = dt;
    const uint32_t raw_row = (uint32_t)r * C::RAW_ROW;
    const uint32_t dst_row = (uint32_t)((r / TC_BM) * TC_TILE_BYTES + (r % TC_BM) * 128);
    const int x7 = r & 7;
    int st_it = 0, raw_it = 0, sl = 0, ph = 0;  // sl, ph: slot and phase of stage st_it
    bool ok = true;
    // the next stage's slot, once the MMAs have released it (false: abort)
    auto stage_begin = [&](int &s) -> bool {
      s = sl;
      return st_it < TC_STAGES || tc_wait(&S.empty[s], ph ^ 1, S, a.status);
    };
    auto stage_end = [&](int s) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.full[s]);
      ++st_it;
      if (++sl == TC_STAGES) sl = 0, ph ^= 1;
    };
    for (int i = 0; ok && bid + G * i < n_tiles; ++i) {
      const TcTile t = tile_of(i);
      const int nk = tile_k<MODE>(a, t) / TC_BK;
      if (t.kind != 0) {  // dense shared-expert tile: its weights come by copy
        for (int kc = 0; ok && kc < nk; ++kc) {
          int s;
          if (!stage_begin(s)) { ok = false; break; }
          stage_end(s);
        }
        continue;
      }
      for (int kb = 0; ok && kb < nk / 4; ++kb) {  // one 256-wide block: four stages
        const int slot = raw_it % TC_RAW_SLOTS;
        if (!tc_wait(&S.raw_full[slot], (raw_it / TC_RAW_SLOTS) & 1, S, a.status)) { ok = false; break; }
        const uint8_t *rb = raw + (size_t)slot * TC_RAW_BYTES + raw_row;
        if (FMT == DS_Q4_K) {
          const uint4 hdr = *reinterpret_cast<const uint4 *>(rb);
          const float d = fp16_to_f32((uint16_t)(hdr.x & 0xFFFFu)), dmin = fp16_to_f32((uint16_t)(hdr.x >> 16));
          for (int q4 = 0; q4 < 4; ++q4) {  // sub-blocks 2 q4 and 2 q4 + 1: eight chunks of the row
            int s;
            if (!stage_begin(s)) { ok = false; break; }
            uint8_t *dst = stages + (size_t)s * TC_STAGE_BYTES + dst_row;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int sb = 2 * q4 + j;
              const float dsc = d * (float)q4k_field(hdr, sb), dmm = dmin * (float)q4k_field(hdr, 8 + sb);  // exact
              uint4 c4[4];
              dequant_q4_sub(*reinterpret_cast<const uint4 *>(rb + 16 + 16 * sb), dsc, dmm, c4);
#pragma unroll
              for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4 *>(dst + (((4 * j + c) ^ x7) << 4)) = c4[c];
            }
            fence_proxy_async();
            stage_end(s);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.raw_empty[slot]);
        } else {
          // The row's 96-byte window in registers with six 16-byte loads (at
          // the 96-byte row pitch these conflict two ways, where word loads
          // conflict eight ways); the raw slot is free once they are done.
          uint32_t W[24];
#pragma unroll
          for (int c = 0; c < 6; ++c) {
            const uint4 v = reinterpret_cast<const uint4 *>(rb)[c];
            W[4 * c] = v.x; W[4 * c + 1] = v.y; W[4 * c + 2] = v.z; W[4 * c + 3] = v.w;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.raw_empty[slot]);
          // the block starts (84 kb) mod 16 bytes = word kb mod 4 into the window
          auto block = [&](auto oc) -> bool {
            constexpr int O = decltype(oc)::value;
            const float d = fp16_to_f32((uint16_t)(W[O + 20] & 0xFFFFu)), dmin = fp16_to_f32((uint16_t)(W[O + 20] >> 16));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {  // quarter of the block in this stage: sub-blocks 4 q4 ..
              int s;
              if (!stage_begin(s)) return false;
              uint8_t *dst = stages + (size_t)s * TC_STAGE_BYTES + dst_row;
              const uint32_t scw = W[O + q4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint4 c0, c1;
                dequant_codes(W[O + 4 + 4 * q4 + j], (scw >> (8 * j)) & 0xFFu, d, dmin, c0, c1);
                *reinterpret_cast<uint4 *>(dst + (((2 * j) ^ x7) << 4)) = c0;
                *reinterpret_cast<uint4 *>(dst + (((2 * j + 1) ^ x7) << 4)) = c1;
              }
              fence_proxy_async();
              stage_end(s);
            }
            return true;
          };
          switch (kb & 3) {
            case 0: ok = block(std::integral_constant<int, 0>()); break;
            case 1: ok = block(std::integral_constant<int, 1>()); break;
            case 2: ok = block(std::integral_constant<int, 2>()); break;
            default: ok = block(std::integral_constant<int, 3>()); break;
          }
        }
        ++raw_it;
      }
    }
  } else if (warp == TC_MMA_WARP) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      // Accumulators: a tile up to 128 tokens wide takes one of the two
      // 256-column buffers in turn (first accumulator at +0, second at +128);
      // a wider one takes both (at 0 and 256).  The epilogue warps walk the
      // same tiles and take the same buffers; fill0 and fill1 count the
      // tiles that each buffer has held, which gives every wait its parity.
      int st_it = 0, sl = 0, ph = 0, nnar = 0, fill0 = 0, fill1 = 0;  // sl, ph: slot and phase of stage st_it
      bool ok = true;
      for (int i = 0; ok && bid + G * i < n_tiles; ++i) {
        const TcTile t = tile_of(i);
        const int K = tile_k<MODE>(a, t), nk = K / TC_BK;
        const int nb = (t.n + 15) & ~15;
        const bool wide = C::A_TILES == 2 && nb > 128;
        const int buf = wide ? 0 : (nnar++ & 1), blast = wide ? 1 : buf;
        bool got = true;
        for (int b = buf; b <= blast; ++b) {
          const int f = b ? fill1 : fill0;
          if (f > 0 && !tc_wait(&S.acc_empty[b], (f & 1) ^ 1, S, a.status)) got = false;
        }
        if (!got) break;
        tc_fence_after();
        const uint32_t idesc = f16_idesc(nb, (GU && t.kind == 1) || MODE == MODE_ROUTER);
        const uint32_t d0 = tmem + (uint32_t)(buf * 256), d1 = d0 + (wide ? 256u : 128u);
        for (int kc = 0; kc < nk; ++kc) {
          const int s = sl;
          if (!tc_wait(&S.full[s], ph, S, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sbase = smem_u32(stages + (size_t)s * TC_STAGE_BYTES);
          const uint32_t bbase = sbase + C::A_TILES * TC_TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t bd = sw128_desc(bbase + 32 * kk);
            if (C::A_TILES == 2) {  // gate and up, or two down blocks: two accumulators
              const bool acc = kc > 0 || kk > 0;
              mma_f16(d0, sw128_desc(sbase + 32 * kk), bd, idesc, acc);
              mma_f16(d1, sw128_desc(sbase + TC_TILE_BYTES + 32 * kk), bd, idesc, acc);
            } else {
              mma_f16(d0, sw128_desc(sbase + 32 * kk), bd, idesc, kc > 0 || kk > 0);
            }
          }
          mma_commit(&S.empty[s]);  // the stage is free once these MMAs have read it
          ++st_it;
          if (++sl == TC_STAGES) sl = 0, ph ^= 1;
        }
        if (!ok) break;
        for (int b = buf; b <= blast; ++b) {
          mma_commit(&S.acc_full[b]);
          (b ? fill1 : fill0) += 1;
        }
      }
      // nothing of this thread may still run when the accumulators are freed
      mma_commit(&S.drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&S.drain, 0))
        if (globaltimer_ns() - t0 > TC_LIMIT_NS) { flag(a.status, ST_TIMEOUT); break; }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue warps --
    const int q = warp;  // TMEM lanes 32 q .. 32 q + 31
    const int r = 32 * q + lane;
    int nnar = 0, fill0 = 0, fill1 = 0;  // the MMA thread's buffer choice, tile by tile
    for (int i = 0; bid + G * i < n_tiles; ++i) {
      const TcTile t = tile_of(i);
      const bool wide = C::A_TILES == 2 && ((t.n + 15) & ~15) > 128;
      const int buf = wide ? 0 : (nnar++ & 1), blast = wide ? 1 : buf;
      bool got = true;
      for (int b = buf; b <= blast; ++b)
        if (!tc_wait(&S.acc_full[b], (b ? fill1 : fill0) & 1, S, a.status)) got = false;
      if (!got) break;
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 256);
      const uint32_t off2 = wide ? 256u : 128u;  // the second accumulator
      if (GU) {
        const int f = t.blk * TC_BM + r;
        const int ld = t.kind == 0 ? a.F : a.Fs;
        // routed h is stored in the permuted K order of the down weights
        uint16_t *hrow = t.kind == 0 ? a.h16 + (int64_t)t.brow * a.F + (f & ~15) + 4 * (f & 3) + ((f & 15) >> 2)
                                     : a.h16 + (int64_t)a.P * a.F + (int64_t)t.brow * a.Fs + f;
        for (int j0 = 0; j0 < t.n; j0 += 16) {
          float g[16], u[16];
          tmem_ld16(tl + j0, g);
          tmem_ld16(tl + off2 + j0, u);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j0 + j < t.n) {
              const float hv = silu(g[j]) * u[j];
              hrow[(int64_t)(j0 + j) * ld] = __half_as_ushort(__float2half_rn(hv));
            }
        }
      } else if (MODE == MODE_ROUTER) {
        const int e = t.blk * TC_BM + r;
        const float b = (a.bias && e < a.E) ? a.bias[e] : 0.f;
        float *orow = a.logits + (int64_t)t.brow * a.E + e;
        for (int j0 = 0; j0 < t.n; j0 += 16) {
          float v[16];
          tmem_ld16(tl + j0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j0 + j < t.n && e < a.E) orow[(int64_t)(j0 + j) * a.E] = v[j] + b;
        }
      } else {
        const int d = 2 * t.blk * TC_BM + r;  // and d + 128 from the second accumulator
        float *orow = (t.kind == 0 ? a.y : a.ys) + (int64_t)t.brow * a.D + d;
        for (int j0 = 0; j0 < t.n; j0 += 16) {
          float v[16], w[16];
          tmem_ld16(tl + j0, v);
          tmem_ld16(tl + off2 + j0, w);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j0 + j < t.n) {
              orow[(int64_t)(j0 + j) * a.D] = v[j];
              orow[(int64_t)(j0 + j) * a.D + TC_BM] = w[j];
            }
        }
      }
      tc_fence_before();
      __syncwarp();
      for (int b = buf; b <= blast; ++b) {
        if (lane == 0) mbar_arrive(&S.acc_empty[b]);
        (b ? fill1 : fill0) += 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS) : "memory");
  }
}

// ------------------------------------------------------------ small kernels --

// Token rows gathered into route order, bf16 -> fp16, each group of 16 in
// the permuted K order: xp[p][16 g + i] = x[perm[p] / k][16 g + 4 (i % 4) + i / 4].
__global__ void __launch_bounds__(256) gather_x16_kernel(const uint16_t *__restrict__ x,
                                                         const int32_t *__restrict__ perm, int64_t P,
                                                         int D, int k, uint16_t *__restrict__ xp,
                                                         unsigned *status) {
  const int ng = D / 16;
  const int64_t n = P * ng;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / ng;
    const int g = (int)(i % ng);
    const int32_t q = perm[p];
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)(q / k) * D + 16 * g);
    const uint4 s0 = src[0], s1 = src[1];
    const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    bool over = false;
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a0 = v[4 * ((2 * j) & 3) + (2 * j) / 4], a1 = v[4 * ((2 * j + 1) & 3) + (2 * j + 1) / 4];
      over |= fabsf(a0) > 65504.f || fabsf(a1) > 65504.f;
      a0 = fminf(fmaxf(a0, -65504.f), 65504.f);
      a1 = fminf(fmaxf(a1, -65504.f), 65504.f);
      const __half2 h = __floats2half2_rn(a0, a1);
      o[j] = *reinterpret_cast<const uint32_t *>(&h);
    }
    if (over) flag(status, ST_RANGE);
    uint4 *dst = reinterpret_cast<uint4 *>(xp + p * D + 16 * g);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// bf16 -> fp16 copy of a matrix (the shared down weights).
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint16_t *__restrict__ src, int64_t n8,
                                                          uint16_t *__restrict__ dst, unsigned *status) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 s = reinterpret_cast<const uint4 *>(src)[i];
    const uint32_t w[4] = {s.x, s.y, s.z, s.w};
    uint32_t o[4];
    bool over = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a0 = __uint_as_float(w[j] << 16), a1 = __uint_as_float(w[j] & 0xFFFF0000u);
      over |= fabsf(a0) > 65504.f || fabsf(a1) > 65504.f;
      a0 = fminf(fmaxf(a0, -65504.f), 65504.f);
      a1 = fminf(fmaxf(a1, -65504.f), 65504.f);
      const __half2 h = __floats2half2_rn(a0, a1);
      o[j] = *reinterpret_cast<const uint32_t *>(&h);
    }
    if (over) flag(status, ST_RANGE);
    reinterpret_cast<uint4 *>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Tile lists of both contractions from the route: shared-expert tiles
// first (full token chunks), then per expert its token chunks times the
// weight-row blocks (chunk-major, so neighbouring tiles share token rows).
// Tokens per tile at most: 128, or with allow_wide 256 when that cuts the
// routed chunks by more than a tenth (experts with more than 128 tokens);
// *wide records the choice for the two GEMM launches, whose ring layout
// follows it.  One block of 1024 threads, one thread per expert.
__global__ void __launch_bounds__(1024) tc_plan_kernel(const int32_t *__restrict__ counts,
                                                       const int32_t *__restrict__ offsets, int E, int64_t T,
                                                       int64_t P, int D, int F, int Fs, int allow_wide,
                                                       int4 *__restrict__ gu, int4 *__restrict__ dn,
                                                       int *__restrict__ n_gu, int *__restrict__ n_dn,
                                                       int *__restrict__ wide) {
  __shared__ int scan_gu[1024], scan_dn[1024];
  __shared__ int n128, n256;
  const int e = threadIdx.x;
  const int ne = e < E ? counts[e] : 0;
  if (e == 0) n128 = n256 = 0;
  __syncthreads();
  if (allow_wide && ne > 0) {
    atomicAdd(&n128, (ne + TC_NGU - 1) / TC_NGU);
    atomicAdd(&n256, (ne + TC_NWIDE - 1) / TC_NWIDE);
  }
  __syncthreads();
  const bool w = allow_wide && 10 * n256 < 9 * n128;
  const int chunk = w ? TC_NWIDE : TC_NGU;
  if (e == 0) *wide = w ? 1 : 0;
  const int cg = (ne + chunk - 1) / chunk, cd = (ne + chunk - 1) / chunk;
  const int tg = cg * (F / TC_BM), td = cd * (D / (2 * TC_BM));
  scan_gu[e] = tg;
  scan_dn[e] = td;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scans
    const int a = e >= o ? scan_gu[e - o] : 0, b = e >= o ? scan_dn[e - o] : 0;
    __syncthreads();
    scan_gu[e] += a;
    scan_dn[e] += b;
    __syncthreads();
  }
  const int sg_chunks = Fs > 0 ? (int)((T + chunk - 1) / chunk) : 0;
  const int sd_chunks = Fs > 0 ? (int)((T + chunk - 1) / chunk) : 0;
  const int n_sg = sg_chunks * (Fs / TC_BM), n_sd = sd_chunks * (D / (2 * TC_BM));
  // shared tiles
  for (int i = e; i < n_sg; i += 1024) {
    const int c = i / (Fs / TC_BM), b = i % (Fs / TC_BM);
    const int t0 = c * chunk, n = (int)min((int64_t)chunk, T - t0);
    gu[i] = make_int4(1, 0, t0, n | (b << 16));
  }
  for (int i = e; i < n_sd; i += 1024) {
    const int c = i / (D / (2 * TC_BM)), b = i % (D / (2 * TC_BM));
    const int t0 = c * chunk, n = (int)min((int64_t)chunk, T - t0);
    dn[i] = make_int4(1, 0, t0, n | (b << 16));
  }
  if (e < E && ne > 0) {
    const int base = offsets[e];
    int o = n_sg + scan_gu[e] - tg;
    for (int c = 0; c < cg; ++c)
      for (int b = 0; b < F / TC_BM; ++b) {
        const int n = min(chunk, ne - c * chunk);
        gu[o++] = make_int4(0, e, base + c * chunk, n | (b << 16));
      }
    o = n_sd + scan_dn[e] - td;
    for (int c = 0; c < cd; ++c)
      for (int b = 0; b < D / (2 * TC_BM); ++b) {
        const int n = min(chunk, ne - c * chunk);
        dn[o++] = make_int4(0, e, base + c * chunk, n | (b << 16));
      }
  }
  if (e == 1023) {
    *n_gu = n_sg + scan_gu[1023];
    *n_dn = n_sd + scan_dn[1023];
  }
}

template <int MODE, int FMT = DS_Q2_K>
constexpr size_t tc_smem() {
  using C = TcCfg<MODE, FMT>;
  return 1024 + C::RING_BYTES + C::RAW * C::RAW_BYTES + sizeof(TcShared);
}
static_assert(tc_smem<MODE_GU>() <= 227 * 1024 && tc_smem<MODE_DN>() <= 227 * 1024 &&
                  tc_smem<MODE_ROUTER>() <= 227 * 1024 && tc_smem<MODE_GU, DS_Q4_K>() <= 227 * 1024 &&
                  tc_smem<MODE_DN, DS_Q4_K>() <= 227 * 1024,
              "pipeline exceeds the shared memory of a block");
static_assert(TcCfg<MODE_DN>::STAGES <= TC_MAX_STAGES && TcCfg<MODE_GU>::RAW <= TC_MAX_RAW, "barrier arrays");

}  // namespace

// ---------------------------------------------------------------- host side --

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major 16-bit matrix [rows][cols] as a 2-D map with 64 x box_rows boxes
// in the 128-byte swizzle (zero fill beyond the edges).
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// The quantised rows of every expert as a 3-D map of 32-bit words: x = word
// in a row, y = row (gate rows then up rows, or down rows), z = expert; boxes
// of box_words words x box_rows rows, no swizzle.
bool make_words_map(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows, int64_t E,
                    int64_t expert_bytes, uint32_t box_words, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)rows, (cuuint64_t)E};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)expert_bytes};
  const cuuint32_t box[3] = {box_words, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_router_tc(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                             cudaStream_t s) {
  static OncePerDevice once;
  const int sms = device_sms();
  if (!sms) return cudaErrorNoDevice;
  const cudaError_t e0 = once_per_device(once, []() {
    return cudaFuncSetAttribute(tc_gemm_kernel<MODE_ROUTER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc_smem<MODE_ROUTER>());
  });
  if (e0 != cudaSuccess) return e0;
  const int64_t T = wk.T;
  TcArgs a{};
  a.D = sh.D; a.F = sh.F; a.Fs = sh.Fs; a.T = (int)T; a.E = sh.E;
  a.router_tiles = (int)(((sh.E + TC_BM - 1) / TC_BM) * ((T + TC_NRT - 1) / TC_NRT));
  a.logits = wk.logits;
  a.bias = W.router_bias;
  a.status = status_word();
  CUtensorMap m_wr, m_x;
  if (!make_map(&m_wr, W.router_w, sh.E, sh.D, TC_BM, true) || !make_map(&m_x, x, T, sh.D, TC_NRT, true))
    return cudaErrorInvalidValue;
  tc_gemm_kernel<MODE_ROUTER><<<std::min<int>(sms, a.router_tiles), TC_THREADS, tc_smem<MODE_ROUTER>(), s>>>(
      a, m_wr, m_x, m_x, m_x, m_x, m_x, m_x, m_x, m_wr, m_wr);
  return cudaGetLastError();
}

bool prefill_tc_supported(const Shape &sh, int64_t T) {
  if (sh.fmt != DS_Q2_K && sh.fmt != DS_Q4_K) return false;
  if (T < TC_MIN_T || T > (int64_t)1 << 24) return false;
  if (sh.x_dtype != DS_BF16 || sh.router_dtype != DS_BF16) return false;
  if (sh.D % 1024 || sh.F % 1024 || sh.Fs % TC_BM) return false;  // whole 4-block groups: raw copies stay inside rows
  if (sh.E > 1024 || T * sh.k > ((int64_t)1 << 31) - 1) return false;
  if ((int64_t)sh.Fs > (int64_t)sh.k * sh.F) return false;  // fp16 h of both kinds fits the fp32 [P][F] region
  return encode_fn() != nullptr;
}

size_t prefill_tc_workspace(const Shape &sh, int64_t T) {
  const int64_t P = T * sh.k;
  const int64_t n_gu = ((T + TC_NGU - 1) / TC_NGU) * (sh.Fs / TC_BM) + (P / TC_NGU + sh.E) * (sh.F / TC_BM);
  const int64_t n_dn = ((T + TC_NDN - 1) / TC_NDN) * (sh.D / TC_BM) + (P / TC_NDN + sh.E) * (sh.D / TC_BM);
  const size_t a = 256;
  auto up = [&](size_t v) { return (v + a - 1) / a * a; };
  return up(2 * (size_t)P * sh.D) + up(2 * (size_t)sh.D * std::max(sh.Fs, 1)) + up(16 * (size_t)n_gu) +
         up(16 * (size_t)n_dn) + up(16);
}

cudaError_t launch_prefill_tc(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                              void *tc_ws, cudaStream_t s) {
  const int64_t T = wk.T, P = T * sh.k;
  unsigned *st = status_word();
  static OncePerDevice once;
  const int sms = device_sms();
  if (!sms) return cudaErrorNoDevice;
  const cudaError_t e0 = once_per_device(once, []() {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_GU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem<MODE_GU>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_DN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem<MODE_DN>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_GU, DS_Q4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tc_smem<MODE_GU, DS_Q4_K>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_DN, DS_Q4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tc_smem<MODE_DN, DS_Q4_K>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_ROUTER>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem<MODE_ROUTER>());
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  const bool q4 = sh.fmt == DS_Q4_K;
  const int64_t bb = sh.block_bytes();
  const uint32_t raw_row = q4 ? TC_RAW_ROW_Q4 : TC_RAW_ROW;
  // workspace carve-up (see prefill_tc_workspace)
  const int64_t n_gu = ((T + TC_NGU - 1) / TC_NGU) * (sh.Fs / TC_BM) + (P / TC_NGU + sh.E) * (sh.F / TC_BM);
  const int64_t n_dn = ((T + TC_NDN - 1) / TC_NDN) * (sh.D / TC_BM) + (P / TC_NDN + sh.E) * (sh.D / TC_BM);
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  char *p = static_cast<char *>(tc_ws);
  uint16_t *xp = reinterpret_cast<uint16_t *>(p);
  p += up(2 * (size_t)P * sh.D);
  uint16_t *sd16 = reinterpret_cast<uint16_t *>(p);
  p += up(2 * (size_t)sh.D * std::max(sh.Fs, 1));
  int4 *tiles_gu = reinterpret_cast<int4 *>(p);
  p += up(16 * (size_t)n_gu);
  int4 *tiles_dn = reinterpret_cast<int4 *>(p);
  p += up(16 * (size_t)n_dn);
  int *cnt = reinterpret_cast<int *>(p);
  uint16_t *h16 = reinterpret_cast<uint16_t *>(wk.h);  // [P + T][F] fp16 fits in the fp32 [P][F] region

  cudaError_t e;
  gather_x16_kernel<<<(unsigned)std::min<int64_t>((P * (sh.D / 16) + 255) / 256, 8 * sms), 256, 0, s>>>(
      (const uint16_t *)x, wk.perm, P, sh.D, sh.k, xp, st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (sh.Fs > 0) {
    const int64_t n8 = (int64_t)sh.D * sh.Fs / 8;
    bf16_to_f16_kernel<<<(unsigned)std::min<int64_t>((n8 + 255) / 256, 8 * sms), 256, 0, s>>>(
        (const uint16_t *)W.shared_down, n8, sd16, st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  tc_plan_kernel<<<1, 1024, 0, s>>>(wk.counts, wk.offsets, sh.E, T, P, sh.D, sh.F, sh.Fs, q4 ? 0 : 1, tiles_gu,
                                    tiles_dn, cnt, cnt + 1, cnt + 2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  TcArgs a{};
  a.D = sh.D; a.F = sh.F; a.Fs = sh.Fs; a.P = (int)P; a.T = (int)T;
  a.experts = W.experts;
  a.expert_bytes = sh.expert_bytes();
  a.gate_bytes = sh.gate_bytes();
  a.h16 = h16;
  a.y = wk.y;
  a.ys = wk.ys;
  a.status = st;
  a.wide = cnt + 2;

  // token boxes of the wide layout (Q2_K): 256 rows; Q4_K has none
  const int wrows = q4 ? TC_NGU : TC_NWIDE;
  CUtensorMap m_xp, m_x, m_xw, m_sg, m_su, m_h, m_sd;
  const int fs1 = std::max(sh.Fs, TC_BM);
  if (!make_map(&m_xp, xp, P, sh.D, wrows, false) || !make_map(&m_x, x, T, sh.D, TC_NGU, true) ||
      !make_map(&m_xw, x, T, sh.D, wrows, true) ||
      !make_map(&m_sg, sh.Fs > 0 ? (const void *)W.shared_gate : (const void *)W.experts, sh.Fs > 0 ? sh.Fs : 1, sh.D, TC_BM, true) ||
      !make_map(&m_su, sh.Fs > 0 ? (const void *)W.shared_up : (const void *)W.experts, sh.Fs > 0 ? sh.Fs : 1, sh.D, TC_BM, true) ||
      !make_map(&m_h, h16, P, sh.F, wrows, false) ||
      !make_map(&m_sd, sd16, sh.D, fs1, TC_BM, false))
    return cudaErrorInvalidValue;
  CUtensorMap m_rgu, m_rdn;
  if (!make_words_map(&m_rgu, W.experts, (int64_t)(sh.D / QK) * bb, 2 * (int64_t)sh.F, sh.E, sh.expert_bytes(), raw_row / 4, TC_BM) ||
      !make_words_map(&m_rdn, W.experts + 2 * sh.gate_bytes(), (int64_t)(sh.F / QK) * bb, sh.D, sh.E,
                      sh.expert_bytes(), raw_row / 4, TC_BM))
    return cudaErrorInvalidValue;
  a.tiles = tiles_gu;
  a.n_tiles = cnt;
  // routed token rows with boxes of 32, 64, 96, 128 and chunk rows
  CUtensorMap m_xp32, m_xp64, m_xp96, m_xp128;
  if (!make_map(&m_xp32, xp, P, sh.D, 32, false) || !make_map(&m_xp64, xp, P, sh.D, 64, false) ||
      !make_map(&m_xp96, xp, P, sh.D, 96, false) || !make_map(&m_xp128, xp, P, sh.D, 128, false))
    return cudaErrorInvalidValue;
  if (q4)
    tc_gemm_kernel<MODE_GU, DS_Q4_K><<<sms, TC_THREADS, tc_smem<MODE_GU, DS_Q4_K>(), s>>>(
        a, m_rgu, m_xp32, m_xp64, m_xp96, m_xp128, m_xp, m_x, m_xw, m_sg, m_su);
  else
    tc_gemm_kernel<MODE_GU><<<sms, TC_THREADS, tc_smem<MODE_GU>(), s>>>(a, m_rgu, m_xp32, m_xp64, m_xp96, m_xp128, m_xp,
                                                                        m_x, m_xw, m_sg, m_su);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the shared rows of h have n_ff_shared columns: their own map
  CUtensorMap m_hs, m_hsw;
  if (!make_map(&m_hs, h16 + (size_t)P * sh.F, T, std::max(sh.Fs, 64), TC_NGU, false) ||
      !make_map(&m_hsw, h16 + (size_t)P * sh.F, T, std::max(sh.Fs, 64), wrows, false))
    return cudaErrorInvalidValue;
  a.tiles = tiles_dn;
  a.n_tiles = cnt + 1;
  CUtensorMap m_h32, m_h64, m_h96, m_h128;
  if (!make_map(&m_h32, h16, P, sh.F, 32, false) || !make_map(&m_h64, h16, P, sh.F, 64, false) ||
      !make_map(&m_h96, h16, P, sh.F, 96, false) || !make_map(&m_h128, h16, P, sh.F, 128, false))
    return cudaErrorInvalidValue;
  if (q4)
    tc_gemm_kernel<MODE_DN, DS_Q4_K><<<sms, TC_THREADS, tc_smem<MODE_DN, DS_Q4_K>(), s>>>(
        a, m_rdn, m_h32, m_h64, m_h96, m_h128, m_h, m_hs, m_hsw, m_sd, m_sd);
  else
    tc_gemm_kernel<MODE_DN><<<sms, TC_THREADS, tc_smem<MODE_DN>(), s>>>(a, m_rdn, m_h32, m_h64, m_h96, m_h128, m_h, m_hs,
                                                                        m_hsw, m_sd, m_sd);
  return cudaGetLastError();
}

}  // namespace dsm
