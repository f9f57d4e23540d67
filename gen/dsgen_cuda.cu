// Device fills of the seeded synthetic-input generator (definition in
// dsgen_core.h).  Produces the same bits as the host fills; used to build
// full-size synthetic layers directly in HBM.  Holds none of the MoE
// method's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>
#include "dsgen_core.h"

namespace {

__global__ void fill_kernel(float *out, uint16_t *out_bf16, uint64_t n, uint32_t seed,
                            uint32_t layer, uint32_t tensor, uint32_t sub, uint64_t idx0,
                            float c, int uniform) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = uniform ? dsgen_uniform(seed, layer, tensor, sub, idx0 + i, c)
                      : dsgen_normal(seed, layer, tensor, sub, idx0 + i, c);
    if (out) out[i] = v;
    if (out_bf16) out_bf16[i] = dsgen_f32_to_bf16(v);
  }
}

__global__ void x_rows_kernel(float *out, uint16_t *out_bf16, int64_t T, int64_t D,
                              const int32_t *attempt, uint32_t seed, uint32_t layer, float c) {
  uint64_t n = (uint64_t)T * (uint64_t)D;
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    int64_t t = (int64_t)(i / (uint64_t)D);
    uint32_t a = attempt ? (uint32_t)attempt[t] : 0u;
    float v = dsgen_normal(seed, layer, DSGEN_T_X, a, i, c);
    if (out) out[i] = v;
    if (out_bf16) out_bf16[i] = dsgen_f32_to_bf16(v);
  }
}

int grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  if (b > 152ull * 64ull) b = 152ull * 64ull;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

extern "C" {

int dsgen_cuda_fill(float *out, uint16_t *out_bf16, uint64_t n, uint32_t seed, uint32_t layer,
                    uint32_t tensor, uint32_t sub, uint64_t idx0, float c, int uniform,
                    cudaStream_t stream) {
  if (n == 0) return 0;
  fill_kernel<<<grid_for(n), 256, 0, stream>>>(out, out_bf16, n, seed, layer, tensor, sub, idx0, c,
                                               uniform);
  return (int)cudaGetLastError();
}

int dsgen_cuda_x_rows(float *out, uint16_t *out_bf16, int64_t T, int64_t D, const int32_t *attempt,
                      uint32_t seed, uint32_t layer, float c, cudaStream_t stream) {
  if (T * D == 0) return 0;
  x_rows_kernel<<<grid_for((uint64_t)(T * D)), 256, 0, stream>>>(out, out_bf16, T, D, attempt, seed,
                                                                 layer, c);
  return (int)cudaGetLastError();
}

}
