// ds_moe_layer_noalloc: the layer with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: plugins inside a host program whose own allocator owns all device
// memory, and latency-critical loops where the implicit device-wide
// synchronisation of cudaMalloc is not acceptable.  For them this entry point
// needs no workspace argument: it uses a fixed array that lives in this
// file's device module, sized NOALLOC_SCRATCH_BYTES.
//
// The array is allocated once per GPU when the library's module is loaded
// there and is held until the process exits.  All calls share it, and it
// keeps the previous call's contents; the layer clears its control words at
// the start of every call, and nothing else in the scratch has to start at
// zero.  Calls whose execution overlaps on the GPU (different streams, or
// several host threads) race on the array and must be serialised by the
// caller.
#include <stdio.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 64u << 20;  // 64 MiB per GPU

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current.
void *scratch_address(char *err, size_t errlen, int *rc) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    if (err && errlen) snprintf(err, errlen, "no usable CUDA device: %s", cudaGetErrorString(e));
    *rc = DS_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      if (err && errlen)
        snprintf(err, errlen, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
      *rc = DS_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int ds_moe_layer_noalloc(const ds_moe_shape *shape, const ds_moe_weights *weights,
                                    const void *x, int64_t T, float *out, void *stream, char *err,
                                    size_t errlen) {
  size_t need = 0;
  int rc = ds_moe_workspace_bytes(shape, T, &need, err, errlen);
  if (rc != DS_OK) return rc;
  if (need > NOALLOC_SCRATCH_BYTES) {
    if (err && errlen)
      snprintf(err, errlen,
               "T=%lld needs %zu bytes of scratch; the static scratch holds %zu bytes "
               "(use ds_moe_layer with a caller workspace, or fewer tokens per call)",
               (long long)T, need, NOALLOC_SCRATCH_BYTES);
    return DS_ERR_INVALID_ARG;
  }
  // ds_moe_layer validates the weights and the other arguments in its own
  // order (T == 0 included); the scratch only has to be addressable
  void *scratch = scratch_address(err, errlen, &rc);
  if (!scratch) return rc;
  return ds_moe_layer(shape, weights, x, T, out, scratch, NOALLOC_SCRATCH_BYTES, nullptr, stream,
                      err, errlen);
}
