// C-ABI entry points of the ds_moe library (declared in include/ds_moe.h):
// argument validation, workspace layout, the per-device status word and the
// dispatch of one routed MoE layer onto the kernels.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsm {

__device__ unsigned g_status_word;

// Slots for the values ds_moe_sync_status takes out of the status word.
constexpr unsigned STATUS_SLOTS = 64;
__device__ unsigned g_status_taken[STATUS_SLOTS];

__global__ void status_take_kernel(unsigned slot) { g_status_taken[slot] = atomicExch(&g_status_word, 0u); }

unsigned *status_word() {
  static std::mutex mu;
  static unsigned *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    addr[dev] = (unsigned *)p;
  }
  return addr[dev];
}

int device_sms() {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms[dev] = 0;
  return sms[dev];
}

namespace {

int fail(char *err, size_t errlen, int code, const char *fmt, ...) {
  if (err && errlen) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(err, errlen, fmt, ap);
    va_end(ap);
  }
  return code;
}

int cuda_fail(char *err, size_t errlen, cudaError_t e, const char *what) {
  return fail(err, errlen, DS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_shape(const ds_moe_shape *s, char *err, size_t errlen, Shape *out) {
  if (!s) return fail(err, errlen, DS_ERR_INVALID_ARG, "shape is NULL");
  if (s->n_embd < 256 || s->n_embd > 8192 || s->n_embd % 256)
    return fail(err, errlen, DS_ERR_UNSUPPORTED, "n_embd=%d: need a multiple of 256 in [256, 8192]",
                s->n_embd);
  if (s->n_expert < 1 || s->n_expert > 1024)
    return fail(err, errlen, DS_ERR_UNSUPPORTED, "n_expert=%d: need 1..1024", s->n_expert);
  if (s->n_ff < 128 || s->n_ff > 8192 || s->n_ff % 128)
    return fail(err, errlen, DS_ERR_UNSUPPORTED, "n_ff=%d: need a multiple of 128 in [128, 8192]",
                s->n_ff);
  if (s->n_ff_shared < 0 || s->n_ff_shared > 8192 || s->n_ff_shared % 128)
    return fail(err, errlen, DS_ERR_UNSUPPORTED,
                "n_ff_shared=%d: need 0 or a multiple of 128 up to 8192", s->n_ff_shared);
  if (s->top_k < 1 || s->top_k > 16 || s->top_k > s->n_expert)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "top_k=%d: need 1..min(n_expert, 16)", s->top_k);
  if ((s->x_dtype != DS_F32 && s->x_dtype != DS_BF16) ||
      (s->router_dtype != DS_F32 && s->router_dtype != DS_BF16))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "x_dtype/router_dtype must be DS_F32 or DS_BF16");
  if (!isfinite(s->routed_scale))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "routed_scale is not finite");
  if (!isfinite(s->logit_scale) || s->logit_scale < 0.f)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "logit_scale must be finite and >= 0");
  if (s->bias_select_only != 0 && s->bias_select_only != 1)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "bias_select_only must be 0 or 1");
  if (s->expert_format != DS_Q2_K && s->expert_format != DS_Q4_K)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "expert_format must be DS_Q2_K or DS_Q4_K");
  *out = Shape{s->n_embd, s->n_expert, s->n_ff, s->n_ff_shared, s->top_k,
               s->x_dtype, s->router_dtype, s->routed_scale,
               s->logit_scale == 0.f ? 1.f : s->logit_scale, s->bias_select_only,
               s->expert_format};
  return DS_OK;
}

constexpr size_t ALIGN = 256;
size_t up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }

// Workspace layout; with base == nullptr only the total is computed.
size_t layout(const Shape &sh, int64_t T, char *base, Work *wk) {
  const int64_t P = T * sh.k;
  const int64_t n_chunks = (P + 1023) / 1024;
  const int64_t xbytes = T * sh.D * (sh.x_dtype == DS_BF16 ? 2 : 4);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char *p = base ? base + off : nullptr;
    off += up(bytes);
    return p;
  };
  Work w{};
  w.ctrl = (unsigned *)take(256);
  w.logits = (float *)take(sizeof(float) * T * sh.E);
  w.ids = (int32_t *)take(sizeof(int32_t) * P);
  w.w = (float *)take(sizeof(float) * P);
  w.counts = (int32_t *)take(sizeof(int32_t) * sh.E);
  w.offsets = (int32_t *)take(sizeof(int32_t) * (sh.E + 1));
  w.perm = (int32_t *)take(sizeof(int32_t) * P);
  w.pos = (int32_t *)take(sizeof(int32_t) * P);
  w.used = (int32_t *)take(sizeof(int32_t) * (sh.E + 1));
  w.chunk = (int32_t *)take(sizeof(int32_t) * n_chunks * sh.E);
  w.h = (float *)take(sizeof(float) * P * sh.F);
  w.hs = (float *)take(sizeof(float) * T * std::max(sh.Fs, 1));
  w.y = (float *)take(sizeof(float) * P * sh.D);
  w.ys = (float *)take(sizeof(float) * T * sh.D);
  w.xn = (uint16_t *)take(sizeof(uint16_t) * T * sh.D);
  w.x_dev = take(xbytes);
  w.out_dev = (float *)take(sizeof(float) * T * sh.D);
  w.tc = prefill_tc_supported(sh, T) ? (void *)take(prefill_tc_workspace(sh, T)) : nullptr;
  w.mt = decode_mt_supported(sh, T) ? (void *)take(decode_mt_workspace(sh, T)) : nullptr;
  if (!base) w.tc = w.mt = nullptr;
  w.T = T;
  w.n_chunks = n_chunks;
  if (wk) *wk = w;
  return off;
}

int check_weights(const Shape &sh, const ds_moe_weights *W, char *err, size_t errlen, bool need_experts = true) {
  if (!W) return fail(err, errlen, DS_ERR_INVALID_ARG, "weights is NULL");
  if (!W->router_w || (need_experts && !W->experts))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "router_w and experts are required");
  if (!aligned(W->router_w, 16) || (W->experts && !aligned(W->experts, 16)))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "router_w / experts must be 16-byte aligned");
  if (W->router_bias && !aligned(W->router_bias, 4))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "router_bias must be 4-byte aligned");
  if (sh.Fs > 0) {
    if (!W->shared_gate || !W->shared_up || !W->shared_down)
      return fail(err, errlen, DS_ERR_INVALID_ARG, "shared expert weights required when n_ff_shared > 0");
    if (!aligned(W->shared_gate, 16) || !aligned(W->shared_up, 16) || !aligned(W->shared_down, 16))
      return fail(err, errlen, DS_ERR_INVALID_ARG, "shared expert weights must be 16-byte aligned");
  }
  return DS_OK;
}

// One layer on device buffers: route, expert FFNs, combine into out.
int run_layer(const Shape &sh, const ds_moe_weights &W, const void *x, float *out, bool accumulate,
              const Work &wk, const ds_moe_debug *dbg, cudaStream_t s, char *err, size_t errlen,
              const Residency *res = nullptr) {
  cudaError_t e;
  // the batched kernels take precedence over the chain where both apply
  const bool mt = !res && wk.mt && aligned(x, 16) && decode_mt_supported(sh, wk.T);
  if (!mt && fused_decode_supported(sh, wk.T)) {
    if ((e = launch_decode_fused(sh, W, x, wk, out, accumulate, s, nullptr, res)) != cudaSuccess)
      return cuda_fail(err, errlen, e, "fused decode layer");
  } else if (res) {  // residency: the kernels that address each expert by pointer
    if ((e = cudaMemsetAsync(wk.ctrl, 0, 256, s)) != cudaSuccess)
      return cuda_fail(err, errlen, e, "workspace control reset");
    if ((e = launch_route(sh, W, x, wk, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "route");
    if ((e = launch_decode_ffn(sh, W, x, wk, s, res)) != cudaSuccess) return cuda_fail(err, errlen, e, "expert FFN");
    if ((e = launch_combine(sh, wk, out, accumulate, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "combine");
  } else if (mt) {
    if ((e = launch_router_logits(sh, W, x, wk, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "router");
    if ((e = launch_decode_mt(sh, W, x, wk, out, accumulate, wk.mt, s)) != cudaSuccess)
      return cuda_fail(err, errlen, e, "batched decode layer");
  } else {
    if ((e = cudaMemsetAsync(wk.ctrl, 0, 256, s)) != cudaSuccess)
      return cuda_fail(err, errlen, e, "workspace control reset");
    if (wk.tc && aligned(x, 16) && prefill_tc_supported(sh, wk.T)) {
      // the router GEMM's tiles hold 256 tokens x 128 experts: below 256
      // tokens it would run on a couple of SMs, so the GEMV router serves
      if (wk.T < 256) {
        if ((e = launch_route(sh, W, x, wk, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "route");
      } else {
        if ((e = launch_router_tc(sh, W, x, wk, s)) != cudaSuccess)
          return cuda_fail(err, errlen, e, "router (tensor cores)");
        if ((e = launch_select_route(sh, wk, W.router_bias, s)) != cudaSuccess)
          return cuda_fail(err, errlen, e, "route");
      }
      if ((e = launch_prefill_tc(sh, W, x, wk, wk.tc, s)) != cudaSuccess)
        return cuda_fail(err, errlen, e, "expert FFN (tensor cores)");
    } else {
      if ((e = launch_route(sh, W, x, wk, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "route");
      if ((e = launch_decode_ffn(sh, W, x, wk, s)) != cudaSuccess) return cuda_fail(err, errlen, e, "expert FFN");
    }
    if ((e = launch_combine(sh, wk, out, accumulate, s)) != cudaSuccess)
      return cuda_fail(err, errlen, e, "combine");
  }
  if (dbg) {
    const int64_t P = wk.T * sh.k;
    struct { void *dst; const void *src; size_t n; } cp[] = {
        {dbg->logits, wk.logits, sizeof(float) * wk.T * sh.E},
        {dbg->ids, wk.ids, sizeof(int32_t) * P},
        {dbg->w, wk.w, sizeof(float) * P},
        {dbg->counts, wk.counts, sizeof(int32_t) * sh.E},
        {dbg->offsets, wk.offsets, sizeof(int32_t) * (sh.E + 1)},
        {dbg->perm, wk.perm, sizeof(int32_t) * P},
    };
    for (auto &c : cp)
      if (c.dst && c.n) {
        e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(err, errlen, e, "debug copy");
      }
  }
  return DS_OK;
}

}  // namespace

int32_t *workspace_counts(const Shape &sh, int64_t T, void *workspace) {
  Work wk;
  layout(sh, T, (char *)workspace, &wk);
  return wk.counts;
}

}  // namespace dsm

using namespace dsm;

extern "C" {

size_t ds_moe_q2k_bytes(int64_t rows, int64_t in_dim) {
  if (rows < 0 || in_dim < 0) return 0;
  return (size_t)rows * (size_t)((in_dim + QK - 1) / QK) * QB;
}

size_t ds_moe_q4k_bytes(int64_t rows, int64_t in_dim) {
  if (rows < 0 || in_dim < 0) return 0;
  return (size_t)rows * (size_t)((in_dim + QK - 1) / QK) * Q4B;
}

size_t ds_moe_expert_bytes(int32_t n_embd, int32_t n_ff) {
  return ds_moe_expert_bytes_fmt(DS_Q2_K, n_embd, n_ff);
}

size_t ds_moe_expert_bytes_fmt(int32_t expert_format, int32_t n_embd, int32_t n_ff) {
  if (n_embd <= 0 || n_ff <= 0) return 0;
  if (expert_format == DS_Q2_K) return 2 * ds_moe_q2k_bytes(n_ff, n_embd) + ds_moe_q2k_bytes(n_embd, n_ff);
  if (expert_format == DS_Q4_K) return 2 * ds_moe_q4k_bytes(n_ff, n_embd) + ds_moe_q4k_bytes(n_embd, n_ff);
  return 0;
}

static int quantize_fmt(int fmt, const float *w, int64_t rows, int64_t in_dim, uint8_t *out,
                        void *stream, char *err, size_t errlen) {
  if (rows < 0 || in_dim < 0) return fail(err, errlen, DS_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || in_dim == 0) return DS_OK;
  if (!w || !out) return fail(err, errlen, DS_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(w, 4) || !aligned(out, 4))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "w and out must be 4-byte aligned");
  if (!status_word()) return fail(err, errlen, DS_ERR_CUDA, "no CUDA device");
  cudaError_t e = launch_quantize(fmt, w, rows, in_dim, out, (cudaStream_t)stream);
  return e == cudaSuccess ? DS_OK : cuda_fail(err, errlen, e, "quantize");
}

static int dequantize_fmt(int fmt, const uint8_t *q, int64_t rows, int64_t in_dim, float *out,
                          void *stream, char *err, size_t errlen) {
  if (rows < 0 || in_dim < 0) return fail(err, errlen, DS_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || in_dim == 0) return DS_OK;
  if (!q || !out) return fail(err, errlen, DS_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(out, 4)) return fail(err, errlen, DS_ERR_INVALID_ARG, "out must be 4-byte aligned");
  cudaError_t e = launch_dequantize(fmt, q, rows, in_dim, out, (cudaStream_t)stream);
  return e == cudaSuccess ? DS_OK : cuda_fail(err, errlen, e, "dequantize");
}

int ds_moe_quantize_q2k(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, void *stream,
                        char *err, size_t errlen) {
  return quantize_fmt(DS_Q2_K, w, rows, in_dim, out, stream, err, errlen);
}

int ds_moe_dequantize_q2k(const uint8_t *q, int64_t rows, int64_t in_dim, float *out, void *stream,
                          char *err, size_t errlen) {
  return dequantize_fmt(DS_Q2_K, q, rows, in_dim, out, stream, err, errlen);
}

int ds_moe_quantize_q4k(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, void *stream,
                        char *err, size_t errlen) {
  return quantize_fmt(DS_Q4_K, w, rows, in_dim, out, stream, err, errlen);
}

int ds_moe_dequantize_q4k(const uint8_t *q, int64_t rows, int64_t in_dim, float *out, void *stream,
                          char *err, size_t errlen) {
  return dequantize_fmt(DS_Q4_K, q, rows, in_dim, out, stream, err, errlen);
}

int ds_moe_workspace_bytes(const ds_moe_shape *shape, int64_t T, size_t *bytes, char *err,
                           size_t errlen) {
  Shape sh{};
  int rc = check_shape(shape, err, errlen, &sh);
  if (rc) return rc;
  if (!bytes) return fail(err, errlen, DS_ERR_INVALID_ARG, "bytes is NULL");
  if (T < 0 || T > (1 << 24)) return fail(err, errlen, DS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  *bytes = layout(sh, T, nullptr, nullptr);
  return DS_OK;
}

int ds_moe_layer(const ds_moe_shape *shape, const ds_moe_weights *weights, const void *x, int64_t T,
                 float *out, void *workspace, size_t workspace_bytes, const ds_moe_debug *dbg,
                 void *stream, char *err, size_t errlen) {
  Shape sh{};
  int rc = check_shape(shape, err, errlen, &sh);
  if (rc) return rc;
  if ((rc = check_weights(sh, weights, err, errlen))) return rc;
  if (T < 0 || T > (1 << 24)) return fail(err, errlen, DS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (T == 0) return DS_OK;
  if (!x || !out || !workspace) return fail(err, errlen, DS_ERR_INVALID_ARG, "x, out and workspace are required");
  if (!aligned(x, 16) || !aligned(out, 16))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  if (!aligned(workspace, ALIGN))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = layout(sh, T, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                workspace_bytes, need);
  if (!status_word()) return fail(err, errlen, DS_ERR_CUDA, "no CUDA device");
  Work wk;
  layout(sh, T, (char *)workspace, &wk);
  return run_layer(sh, *weights, x, out, false, wk, dbg, (cudaStream_t)stream, err, errlen);
}

// The device address of host memory, or null if the device cannot address it.
static void *device_view(const void *host) {
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, host) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if ((pa.type == cudaMemoryTypeHost || pa.type == cudaMemoryTypeManaged) && pa.devicePointer) return pa.devicePointer;
  return nullptr;
}

int ds_moe_layer_hostio(const ds_moe_shape *shape, const ds_moe_weights *weights,
                        const void *x_host, int64_t T, float *out_host, void *workspace,
                        size_t workspace_bytes, void *stream, char *err, size_t errlen) {
  Shape sh{};
  int rc = check_shape(shape, err, errlen, &sh);
  if (rc) return rc;
  if ((rc = check_weights(sh, weights, err, errlen))) return rc;
  if (T < 0 || T > (1 << 24)) return fail(err, errlen, DS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (T == 0) return DS_OK;
  if (!x_host || !out_host || !workspace)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "x_host, out_host and workspace are required");
  if (!aligned(workspace, ALIGN))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = layout(sh, T, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                workspace_bytes, need);
  if (!status_word()) return fail(err, errlen, DS_ERR_CUDA, "no CUDA device");
  Work wk;
  layout(sh, T, (char *)workspace, &wk);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t xbytes = (size_t)T * sh.D * (sh.x_dtype == DS_BF16 ? 2 : 4);
  // one token in host memory the device can address (pinned, or any memory
  // on a coherent host): the kernels read x and write out there directly,
  // with one device copy of x made by the router grid; no copy operations
  if (fused_decode_supported(sh, T) && stream_decode_supported(sh, T)) {
    const void *xd = device_view(x_host);
    void *od = device_view(out_host);
    if (xd && od && aligned(xd, 16)) {
      cudaError_t ed = launch_decode_fused(sh, *weights, xd, wk, (float *)od, false, s, wk.x_dev);
      return ed == cudaSuccess ? DS_OK : cuda_fail(err, errlen, ed, "fused decode layer (host buffers)");
    }
  }
  cudaError_t e = cudaMemcpyAsync(wk.x_dev, x_host, xbytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(err, errlen, e, "copy x to device");
  rc = run_layer(sh, *weights, wk.x_dev, wk.out_dev, false, wk, nullptr, s, err, errlen);
  if (rc) return rc;
  e = cudaMemcpyAsync(out_host, wk.out_dev, sizeof(float) * T * sh.D, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? DS_OK : cuda_fail(err, errlen, e, "copy out to host");
}

// Checks a residency view and turns it into the kernels' form (device view of
// the host copy).
static int residency_of(const Shape &sh, const ds_moe_residency *r, Residency *out, char *err, size_t errlen) {
  if (!r) return fail(err, errlen, DS_ERR_INVALID_ARG, "residency is NULL");
  if (!r->slot || !r->experts_host)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "residency needs a slot table and the host copy of the experts");
  if (!aligned(r->slot, 4) || (r->cache && !aligned(r->cache, 16)))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "slot table must be 4-byte and cache 16-byte aligned");
  const void *hv = device_view(r->experts_host);
  if (!hv || !aligned(hv, 16))
    return fail(err, errlen, DS_ERR_INVALID_ARG,
                "experts_host must be 16-byte aligned host memory the device can address (pinned or registered)");
  (void)sh;
  *out = Residency{r->slot, r->cache, (const uint8_t *)hv};
  return DS_OK;
}

int ds_moe_layer_resident(const ds_moe_shape *shape, const ds_moe_weights *weights,
                          const ds_moe_residency *residency, const void *x, int64_t T, float *out,
                          void *workspace, size_t workspace_bytes, const ds_moe_debug *dbg, void *stream,
                          char *err, size_t errlen) {
  Shape sh{};
  int rc = check_shape(shape, err, errlen, &sh);
  if (rc) return rc;
  if ((rc = check_weights(sh, weights, err, errlen, false))) return rc;
  Residency res{};
  if ((rc = residency_of(sh, residency, &res, err, errlen))) return rc;
  if (T < 0 || T > (1 << 24)) return fail(err, errlen, DS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (T == 0) return DS_OK;
  if (!x || !out || !workspace) return fail(err, errlen, DS_ERR_INVALID_ARG, "x, out and workspace are required");
  if (!aligned(x, 16) || !aligned(out, 16))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  if (!aligned(workspace, ALIGN))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = layout(sh, T, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  if (!status_word()) return fail(err, errlen, DS_ERR_CUDA, "no CUDA device");
  Work wk;
  layout(sh, T, (char *)workspace, &wk);
  return run_layer(sh, *weights, x, out, false, wk, dbg, (cudaStream_t)stream, err, errlen, &res);
}

int ds_moe_stack_mixed(const ds_moe_shape *shape, const ds_moe_weights *layers,
                       const int32_t *formats, int32_t n_layers, float *x, int64_t T, float eps,
                       void *workspace, size_t workspace_bytes, void *stream, char *err,
                       size_t errlen) {
  Shape sh{};
  int rc = check_shape(shape, err, errlen, &sh);
  if (rc) return rc;
  if (sh.x_dtype != DS_BF16)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "the stack feeds bf16 normalised inputs: x_dtype must be DS_BF16");
  if (n_layers < 0 || (n_layers > 0 && !layers))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "bad layer array");
  // the workspace serves every layer: laid out for Q2_K when any layer is
  // Q2_K (its tensor-core scratch comes last and the other regions do not
  // depend on the format)
  bool any_q2 = false;
  for (int l = 0; l < n_layers; ++l) {
    const int f = formats ? formats[l] : sh.fmt;
    if (f != DS_Q2_K && f != DS_Q4_K)
      return fail(err, errlen, DS_ERR_INVALID_ARG, "formats[%d]=%d: need DS_Q2_K or DS_Q4_K", l, f);
    any_q2 = any_q2 || f == DS_Q2_K;
  }
  Shape sh_ws = sh;
  sh_ws.fmt = any_q2 ? DS_Q2_K : DS_Q4_K;
  for (int l = 0; l < n_layers; ++l)
    if ((rc = check_weights(sh, &layers[l], err, errlen))) return rc;
  if (T < 0 || T > (1 << 24)) return fail(err, errlen, DS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (T == 0 || n_layers == 0) return DS_OK;
  if (!x || !workspace) return fail(err, errlen, DS_ERR_INVALID_ARG, "x and workspace are required");
  if (!aligned(x, 16) || !aligned(workspace, ALIGN))
    return fail(err, errlen, DS_ERR_INVALID_ARG, "x must be 16-byte and workspace 256-byte aligned");
  if (!(eps > 0.0f) || !isfinite(eps)) return fail(err, errlen, DS_ERR_INVALID_ARG, "eps must be > 0");
  const size_t need = layout(sh_ws, T, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(err, errlen, DS_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                workspace_bytes, need);
  if (!status_word()) return fail(err, errlen, DS_ERR_CUDA, "no CUDA device");
  Work wk;
  layout(sh_ws, T, (char *)workspace, &wk);
  cudaStream_t s = (cudaStream_t)stream;
  for (int l = 0; l < n_layers; ++l) {
    Shape sl = sh;
    if (formats) sl.fmt = formats[l];
    cudaError_t e = launch_rmsnorm_bf16(x, T, sh.D, eps, wk.xn, s);
    if (e != cudaSuccess) return cuda_fail(err, errlen, e, "rmsnorm");
    rc = run_layer(sl, layers[l], wk.xn, x, true, wk, nullptr, s, err, errlen);
    if (rc) return rc;
  }
  return DS_OK;
}

int ds_moe_stack(const ds_moe_shape *shape, const ds_moe_weights *layers, int32_t n_layers,
                 float *x, int64_t T, float eps, void *workspace, size_t workspace_bytes,
                 void *stream, char *err, size_t errlen) {
  return ds_moe_stack_mixed(shape, layers, nullptr, n_layers, x, T, eps, workspace,
                            workspace_bytes, stream, err, errlen);
}

int ds_moe_sync_status(void *stream, char *err, size_t errlen) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(err, errlen, e, "stream");
  // read and clear in one atomic exchange on the device, so that bits another
  // stream's kernel sets meanwhile are kept for the next call; each call
  // takes its own slot for the value read
  static std::atomic<unsigned> next_slot{0};
  const unsigned slot = next_slot.fetch_add(1u) % STATUS_SLOTS;
  status_take_kernel<<<1, 1, 0, s>>>(slot);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, errlen, e, "status exchange");
  unsigned v = 0;
  e = cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof v, sizeof(unsigned) * slot, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(err, errlen, e, "read status word");
  if (v & ST_TIMEOUT) return fail(err, errlen, DS_ERR_TIMEOUT, "a device wait timed out (status 0x%x)", v);
  if (v & ST_QUANT_INPUT)
    return fail(err, errlen, DS_ERR_DEVICE_CHECK, "quantiser input not finite or |w| > 65504 (status 0x%x)", v);
  if (v & ST_BAD_ID)
    return fail(err, errlen, DS_ERR_DEVICE_CHECK,
                "a token with fewer than top_k non-NaN router logits, or an expert id out of range (status 0x%x)", v);
  if (v & ST_RANGE)
    return fail(err, errlen, DS_ERR_DEVICE_CHECK,
                "a value beyond the fp16 range reached the tensor-core path and was saturated (status 0x%x)", v);
  if (v) return fail(err, errlen, DS_ERR_DEVICE_CHECK, "device check failed (status 0x%x)", v);
  return DS_OK;
}

int ds_moe_layer_path(const ds_moe_shape *shape, int64_t T, const void *x) {
  Shape sh;
  if (check_shape(shape, nullptr, 0, &sh) != DS_OK || T < 0) return DS_ERR_INVALID_ARG;
  if (T == 0) return DS_PATH_NONE;
  if (aligned(x, 16) && decode_mt_supported(sh, T)) return DS_PATH_BATCHED_DECODE;
  if (fused_decode_supported(sh, T)) return stream_decode_supported(sh, T) ? DS_PATH_STREAM : DS_PATH_DECODE3;
  if (aligned(x, 16) && prefill_tc_supported(sh, T)) return DS_PATH_TENSOR_CORE;
  return DS_PATH_GROUPED_GEMV;
}

int ds_moe_layer_path_resident(const ds_moe_shape *shape, int64_t T) {
  Shape sh;
  if (check_shape(shape, nullptr, 0, &sh) != DS_OK || T < 0) return DS_ERR_INVALID_ARG;
  if (T == 0) return DS_PATH_NONE;
  if (fused_decode_supported(sh, T)) return stream_decode_supported(sh, T) ? DS_PATH_STREAM : DS_PATH_DECODE3;
  return DS_PATH_GROUPED_GEMV;
}

const char *ds_moe_version(void) { return "ds_moe 0.2 (sm_103a)"; }

}  // extern "C"
