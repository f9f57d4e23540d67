// Shared device helpers of the ds_moe CUDA library (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds_moe.h"

namespace dsm {

constexpr int QK = 256;      // weights per Q2_K super-block
constexpr int QB = 84;       // bytes per Q2_K super-block
constexpr int Q4B = 144;     // bytes per Q4_K super-block
constexpr int NUM_SMS = 152; // GB300

// Sticky status bits (per device, read by ds_moe_sync_status).
enum : unsigned {
  ST_QUANT_INPUT = 1u << 0,   // non-finite / out-of-range quantiser input
  ST_BAD_ID = 1u << 1,        // expert id outside [0, E), or a pick with no candidate (NaN logits)
  ST_TIMEOUT = 1u << 2,       // a bounded device wait expired
  ST_BAD_COUNT = 1u << 3,     // route counts inconsistent
  ST_RANGE = 1u << 4,         // a value beyond the fp16 range met the tensor-core path (saturated)
};

// Status word address for the current device (set up once per device).
unsigned *status_word();

__device__ __forceinline__ void flag(unsigned *st, unsigned bit) { atomicOr(st, bit); }

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float fp16_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

// 6-bit field i of a Q4_K block header h (its first 16 bytes: fp16 d and
// dmin, then the fields as one 96-bit little-endian integer, field i in bits
// [6 i, 6 i + 6); fields 0..7 are the sub-block scales, 8..15 the mins).
__device__ __forceinline__ int q4k_field(const uint4 &h, int i) {
  const uint64_t lo = (uint64_t)h.y | ((uint64_t)h.z << 32);
  const int p = 6 * i;
  if (p + 6 <= 64) return (int)((lo >> p) & 63u);
  if (p >= 64) return (int)((h.w >> (p - 64)) & 63u);
  return (int)(((lo >> p) | ((uint64_t)h.w << (64 - p))) & 63u);
}

// fp32 -> unsigned key with the same order (for non-NaN values), and back.
__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ----------------------------------------------------------------------------
// Host-side launch helpers
// ----------------------------------------------------------------------------

struct Shape {
  int D, E, F, Fs, k;
  int x_dtype, router_dtype;
  float routed_scale;
  float logit_scale;  // 1: plain softmax over the selected logits
  int bias_select_only;  // 1: the router bias steers the selection only
  int fmt;               // ds_expert_format of the routed experts
  int block_bytes() const { return fmt == DS_Q4_K ? Q4B : QB; }
  int64_t nb_D() const { return (D + QK - 1) / QK; }
  int64_t nb_F() const { return (F + QK - 1) / QK; }
  int64_t gate_bytes() const { return (int64_t)F * nb_D() * block_bytes(); }
  int64_t down_bytes() const { return (int64_t)D * nb_F() * block_bytes(); }
  int64_t expert_bytes() const { return 2 * gate_bytes() + down_bytes(); }
};

}  // namespace dsm
