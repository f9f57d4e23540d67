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
  int my_id = 0;
  float my_v = 0.f;
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

}  // namespace
}  // namespace dsm
