// Internal launchers of the ds_moe library (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace dsm {

// Device views of the per-call workspace (all device pointers).
struct Work {
  float *logits;     // [T][E]
  int32_t *ids;      // [T][k]
  float *w;          // [T][k]
  int32_t *counts;   // [E]
  int32_t *offsets;  // [E+1]
  int32_t *perm;     // [T*k]
  int32_t *pos;      // [T*k]
  int32_t *used;     // [E+1]: used[0..n) ascending experts with tokens, used[E] = n
  int32_t *chunk;    // [n_chunks][E] per-chunk histogram (large T)
  unsigned *ctrl;    // control words (zeroed at the start of every call)
  float *h;          // [T*k][F] routed SwiGLU activations, perm order
  float *hs;         // [T][Fs] shared-expert activations
  float *y;          // [T*k][D] routed expert outputs, perm order
  float *ys;         // [T][D] shared-expert output
  uint16_t *xn;      // [T][D] bf16 normalised input (stack)
  void *x_dev;       // [T][D] device copy of host x (hostio)
  float *out_dev;    // [T][D] device out (hostio)
  void *tc;          // tensor-core path scratch (prefill_tc_workspace bytes), or null
  void *mt;          // batched decode scratch (decode_mt_workspace bytes), or null
  int64_t T;
  int64_t n_chunks;
};

// Tensor maps for the bulk-tensor (TMA) copies, encoded through the driver
// entry point (null when the driver has none).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();
// Row-major 16-bit matrix [rows][cols] as a 2-D map with boxes of 64 columns
// x box_rows rows in the 128-byte swizzle (zero fill beyond the edges).
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows, bool bf16);
// Quantised expert rows as a 3-D map of 32-bit words {row words, rows, E}.
bool make_words_map(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows, int64_t E,
                    int64_t expert_bytes, uint32_t box_words, uint32_t box_rows);

// The current device's SM count (looked up once per device); 0 without a
// usable device.
int device_sms();

// Per-device one-time set-up of a launch site (kernel attributes): init()
// runs once per device, under a lock, with that device current; later calls
// on the same device return its result.
struct OncePerDevice {
  std::mutex mu;
  signed char state[64] = {};  // 0: not run, 1: done
  cudaError_t err[64] = {};
};
template <class F>
cudaError_t once_per_device(OncePerDevice &o, F &&init) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(o.mu);
  if (!o.state[dev]) {
    o.err[dev] = init();
    o.state[dev] = 1;
  }
  return o.err[dev];
}

// Expert residency of one layer call: slot[e] >= 0 puts expert e in cache
// slot slot[e], -1 in the device view `host` of the host copy of all experts.
struct Residency {
  const int32_t *slot;
  const uint8_t *cache;
  const uint8_t *host;
};

// The per-expert token counts region of a workspace laid out for T tokens.
int32_t *workspace_counts(const Shape &sh, int64_t T, void *workspace);

// fmt: DS_Q2_K or DS_Q4_K.
cudaError_t launch_quantize(int fmt, const float *w, int64_t rows, int64_t in_dim, uint8_t *out,
                            cudaStream_t s);
cudaError_t launch_dequantize(int fmt, const uint8_t *q, int64_t rows, int64_t in_dim, float *out,
                              cudaStream_t s);

// Router logits, top-k selection and the expert route (histogram, scan,
// stable permutation, used-expert list).
cudaError_t launch_route(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                         cudaStream_t s);
// The part of launch_route after the logits: selection and route.
// bias: the router bias the logits include (or null); with
// sh.bias_select_only it is taken back out of the selected logits before the
// softmax of the weights.
cudaError_t launch_select_route(const Shape &sh, const Work &wk, const float *bias, cudaStream_t s);

// Decode path: grouped dequantising GEMVs and the combine.
cudaError_t launch_decode_ffn(const Shape &sh, const ds_moe_weights &W, const void *x,
                              const Work &wk, cudaStream_t s, const Residency *res = nullptr);
// Decode path for T <= 8: the whole layer in one persistent kernel (writes or
// accumulates into out, and fills the route arrays of the workspace).
bool fused_decode_supported(const Shape &sh, int64_t T);
// ... and within it, the one-token streaming kernel.
bool stream_decode_supported(const Shape &sh, int64_t T);
// x_stage (one token, streaming kernel only): x is host memory the device can
// read; the router grid copies it there once and the streaming kernel reads
// the copy.
cudaError_t launch_decode_fused(const Shape &sh, const ds_moe_weights &W, const void *x,
                                const Work &wk, float *out, bool accumulate, cudaStream_t s,
                                void *x_stage = nullptr, const Residency *res = nullptr);
// Large batches: the expert FFNs as grouped tcgen05 GEMMs (after
// launch_route; the combine follows).  tc_ws holds prefill_tc_workspace bytes.
constexpr int64_t TC_MIN_T = 5;
bool prefill_tc_supported(const Shape &sh, int64_t T);
size_t prefill_tc_workspace(const Shape &sh, int64_t T);
cudaError_t launch_prefill_tc(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                              void *tc_ws, cudaStream_t s);
// Router logits of the tensor-core path (bf16 x and router, tcgen05).
cudaError_t launch_router_tc(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                             cudaStream_t s);
// Batched decode (MT_MIN_T..MT_MAX_T tokens): the router logits alone, then
// selection, route, expert FFNs and combine in the batched decode kernels.
// (The kernels hold up to 32 tokens; above 16 the tensor-core path is faster,
// below 4 the three-kernel chain.)
constexpr int64_t MT_MIN_T = 4, MT_MAX_T = 16;
cudaError_t launch_router_logits(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk,
                                 cudaStream_t s);
bool decode_mt_supported(const Shape &sh, int64_t T);
size_t decode_mt_workspace(const Shape &sh, int64_t T);
cudaError_t launch_decode_mt(const Shape &sh, const ds_moe_weights &W, const void *x, const Work &wk, float *out,
                             bool accumulate, void *mt_ws, cudaStream_t s);
cudaError_t launch_combine(const Shape &sh, const Work &wk, float *out, bool accumulate,
                           cudaStream_t s);

// Stack helper: bf16(x / sqrt(mean(x^2) + eps)).
cudaError_t launch_rmsnorm_bf16(const float *x, int64_t T, int D, float eps, uint16_t *out,
                                cudaStream_t s);

}  // namespace dsm
