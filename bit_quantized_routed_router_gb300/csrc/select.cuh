// Top-k selection of one token's router logits by one warp ("Understanding
// Dwarf Star", 5.3.2 "The MoE Architecture": the top-k experts by router
// probability, weighted by it; ties go to the lower expert index).  Shared by
// the route kernels and the batched decode kernels.
#pragma once
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace dsm {
namespace {

// Top-k picks of one token's logits when every lane holds at most eight of
// them (E <= 256; element lane + 32 i in lv[i]).  Each lane first sorts its
// eight candidates (Batcher's odd-even merge network: 19 compare-exchanges,
// larger logit first, then the lower index); a pick is then the warp's
// largest head key and the lowest index holding it (two hardware
// reductions), and the lane that supplied it shifts its list by one, so no
// pick waits on a rescan.  NaN logits are never picked; when fewer than k
// candidates remain the pick is flagged ST_BAD_ID and taken as expert 0.
// Lane lane0 + j (j < k) ends with pick j in (my_id, my_v).  Same picks, in
// the same order, as a scan over all E logits.
__device__ __forceinline__ void topk_sorted8(const float lv[8], int E, int k, int &my_id, float &my_v,
                                             unsigned *st, int lane0 = 0) {
  const int lane = threadIdx.x & 31;
  uint32_t kk[8];
  int id[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    const bool ok = e < E && !isnan(lv[i]);
    kk[i] = ok ? ord_key(lv[i] + 0.f) : 0u;  // -0 as +0: equal logits tie; 0: no candidate
    id[i] = ok ? e : 0x7fffffff;
  }
  constexpr int NET[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6}, {5, 7}, {1, 2}, {5, 6},
                              {0, 4}, {1, 5}, {2, 6}, {3, 7}, {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const int p = NET[c][0], q = NET[c][1];
    const bool sw = kk[q] > kk[p] || (kk[q] == kk[p] && id[q] < id[p]);
    const uint32_t k0 = kk[p], k1 = kk[q];
    const int i0 = id[p], i1 = id[q];
    kk[p] = sw ? k1 : k0; kk[q] = sw ? k0 : k1;
    id[p] = sw ? i1 : i0; id[q] = sw ? i0 : i1;
  }
  for (int j = 0; j < k; ++j) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, kk[0]);
    int wi = (int)__reduce_min_sync(0xffffffffu, kk[0] == mk ? (uint32_t)id[0] : 0x7fffffffu);
    const bool mine = id[0] == wi && kk[0] == mk;
    if (mk == 0u || wi < 0 || wi >= E) {  // no candidate left (NaN logits, or k > E)
      if (lane == 0) flag(st, ST_BAD_ID);
      wi = 0;
    }
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      kk[i] = mine ? kk[i + 1] : kk[i];
      id[i] = mine ? id[i + 1] : id[i];
    }
    kk[7] = mine ? 0u : kk[7];
    id[7] = mine ? 0x7fffffff : id[7];
    if (lane == lane0 + j) { my_id = wi; my_v = ord_val(mk); }
  }
}

// Weights of one token's picks (lane j holds pick j) and the stores.
__device__ __forceinline__ void finish_token(int my_id, float my_v, int k, float routed_scale, float logit_scale,
                                             const float *__restrict__ unbias, int32_t *ids, float *w) {
  const int lane = threadIdx.x & 31;
  if (unbias && lane < k) my_v -= unbias[my_id];
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? __expf(logit_scale * (my_v - m)) : 0.f;
  float den = 0.0f;  // summed in pick order
  for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = routed_scale * (ex / den);
  }
}

// Top-k of one token's logits in the calling warp: ids in descending logit
// order, ties to the lower index; weights = routed_scale * softmax over
// logit_scale * the selected logits, from which `unbias` (the router bias,
// when it steers the selection only; else null) is taken back out.
// E <= 1024, k <= 16.  The lane's logits (elements lane + 32 i) are loaded
// into registers, all loads issued before the first use; lane j ends with
// pick j and writes ids[j], w[j].
__device__ void select_token(const float *__restrict__ L, int E, int k, float routed_scale, float logit_scale,
                             const float *__restrict__ unbias, int32_t *ids, float *w, unsigned *st) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) / 32;
  float lv[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) lv[i] = i < nv && lane + 32 * i < E ? L[lane + 32 * i] : -INFINITY;
  int my_id = 0;
  float my_v = 0.f;
  if (E <= 256) {
    topk_sorted8(lv, E, k, my_id, my_v, st);
    finish_token(my_id, my_v, k, routed_scale, logit_scale, unbias, ids, w);
    return;
  }
  uint32_t taken = 0;  // bit i: element lane + 32 i already selected
  // each lane's best remaining candidate; a pick is the warp's largest
  // order-preserving key (two hardware reductions: the key, then the lowest
  // index holding it), and only the lane that supplied it rescans
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  auto rescan = [&]() {
    bv = -INFINITY;
    bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i >= nv) break;
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && (lv[i] > bv || (lv[i] == bv && e < bi))) { bv = lv[i]; bi = e; }
    }
  };
  rescan();
  for (int j = 0; j < k; ++j) {
    const uint32_t key = ord_key(bv + 0.f);  // -0 as +0: equal logits tie
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
    int wi = (int)__reduce_min_sync(0xffffffffu, key == mk ? (uint32_t)bi : 0x7fffffffu);
    if (wi < 0 || wi >= E) {  // only possible with NaN logits
      if (lane == 0) flag(st, ST_BAD_ID);
      wi = 0;
    }
    if ((wi & 31) == lane && wi == bi) {
      taken |= 1u << (wi >> 5);
      rescan();
    }
    if (lane == j) { my_id = wi; my_v = ord_val(mk); }
  }
  finish_token(my_id, my_v, k, routed_scale, logit_scale, unbias, ids, w);
}

}  // namespace
}  // namespace dsm
