// Expert residency beyond HBM: a cache of routed experts in device memory,
// the rest read from the host copy.
//
// "The sparsity that pays for everything else in DwarfStar" ("Page the
// experts off the SSD", "The cache is never allowed to become a correctness
// structure"): the engine keeps the dense weights resident and pages routed
// experts in through a cache, and the output stays the same whatever the
// cache holds, because the kernels read the same bytes either way.  Here the
// experts live in host memory the GPU can address (on a Grace-Blackwell
// system, read over NVLink-C2C) and a caller-owned pool of device slots
// holds the most recently used ones.  Every layer call reads each expert from
// its slot when it has one and from the host copy otherwise (the same
// kernels, the same bytes), then the experts the call missed are copied into
// free or least recently used slots for the calls that follow.
#include <string.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct ds_moe_cache {
  dsm::Shape sh{};
  int32_t n_layers = 0, E = 0;
  int64_t eb = 0, n_slots = 0;
  std::vector<const uint8_t *> host;  // per layer: the host copy (host pointers, for the fills)
  uint8_t *slots = nullptr;           // device: n_slots experts
  int32_t *tables = nullptr;          // device: [n_layers][E] slot tables (null: planning only)
  std::vector<int32_t> table;         // host mirror of the slot tables
  std::vector<int32_t> owner_layer, owner_e;  // per slot: the expert it holds, or -1
  std::vector<uint64_t> last;         // per slot: the call that last used it
  uint64_t tick = 0;
  int64_t hits = 0, misses = 0;
  mutable std::mutex mu;

  // The experts a call of `layer` used (counts[e] > 0): hits refresh their
  // slots; each miss takes a free slot, else the least recently used slot
  // that this call did not use (none left: it stays in host memory).
  // Appends (slot, expert) fills and marks the layers whose tables changed.
  void record(int32_t layer, const int32_t *counts, std::vector<int32_t> &fills, std::vector<char> &changed) {
    ++tick;
    int32_t *tl = table.data() + (size_t)layer * E;
    std::vector<int32_t> want;
    for (int32_t e = 0; e < E; ++e) {
      if (counts[e] <= 0) continue;
      if (tl[e] >= 0) {
        ++hits;
        last[tl[e]] = tick;
      } else {
        ++misses;
        want.push_back(e);
      }
    }
    for (int32_t e : want) {
      int64_t pick = -1;
      for (int64_t s = 0; s < n_slots; ++s)
        if (owner_e[s] < 0) { pick = s; break; }
      if (pick < 0)
        for (int64_t s = 0; s < n_slots; ++s)
          if (last[s] < tick && (pick < 0 || last[s] < last[pick])) pick = s;
      if (pick < 0) break;  // every slot holds an expert this call used
      if (owner_e[pick] >= 0) {
        table[(size_t)owner_layer[pick] * E + owner_e[pick]] = -1;
        changed[owner_layer[pick]] = 1;
      }
      owner_layer[pick] = layer;
      owner_e[pick] = e;
      last[pick] = tick;
      tl[e] = (int32_t)pick;
      changed[layer] = 1;
      fills.push_back((int32_t)pick);
      fills.push_back(e);
    }
  }
};

namespace {

int cfail(char *err, size_t errlen, int code, const char *msg) {
  if (err && errlen) {
    strncpy(err, msg, errlen - 1);
    err[errlen - 1] = 0;
  }
  return code;
}

}  // namespace

extern "C" {

int ds_moe_cache_create(const ds_moe_shape *shape, int32_t n_layers, const void *const *experts_host,
                        void *slots, int64_t n_slots, int32_t *tables, ds_moe_cache **cache, char *err,
                        size_t errlen) {
  if (!cache) return cfail(err, errlen, DS_ERR_INVALID_ARG, "cache is NULL");
  *cache = nullptr;
  size_t ws = 0;
  int rc = ds_moe_workspace_bytes(shape, 1, &ws, err, errlen);  // validates the shape
  if (rc) return rc;
  if (n_layers < 1 || n_slots < 0) return cfail(err, errlen, DS_ERR_INVALID_ARG, "n_layers >= 1 and n_slots >= 0");
  if (!experts_host) return cfail(err, errlen, DS_ERR_INVALID_ARG, "experts_host is NULL");
  for (int32_t l = 0; l < n_layers; ++l)
    if (!experts_host[l]) return cfail(err, errlen, DS_ERR_INVALID_ARG, "a layer's host experts are NULL");
  if (tables && n_slots > 0 && !slots)
    return cfail(err, errlen, DS_ERR_INVALID_ARG, "slots are required when the cache holds experts");
  if ((slots && (uintptr_t)slots % 16) || (tables && (uintptr_t)tables % 4))
    return cfail(err, errlen, DS_ERR_INVALID_ARG, "slots must be 16-byte and tables 4-byte aligned");
  ds_moe_cache *c = new ds_moe_cache();
  c->sh = dsm::Shape{shape->n_embd, shape->n_expert, shape->n_ff, shape->n_ff_shared, shape->top_k,
                     shape->x_dtype, shape->router_dtype, shape->routed_scale, shape->logit_scale,
                     shape->bias_select_only, shape->expert_format};
  c->n_layers = n_layers;
  c->E = shape->n_expert;
  c->eb = (int64_t)ds_moe_expert_bytes_fmt(shape->expert_format, shape->n_embd, shape->n_ff);
  c->n_slots = n_slots;
  for (int32_t l = 0; l < n_layers; ++l) c->host.push_back((const uint8_t *)experts_host[l]);
  c->slots = (uint8_t *)slots;
  c->tables = tables;
  c->table.assign((size_t)n_layers * c->E, -1);
  c->owner_layer.assign((size_t)n_slots, -1);
  c->owner_e.assign((size_t)n_slots, -1);
  c->last.assign((size_t)n_slots, 0);
  if (tables) {  // every expert starts in host memory
    const cudaError_t e = cudaMemcpy(tables, c->table.data(), sizeof(int32_t) * c->table.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      delete c;
      return cfail(err, errlen, DS_ERR_CUDA, cudaGetErrorString(e));
    }
  }
  *cache = c;
  return DS_OK;
}

void ds_moe_cache_destroy(ds_moe_cache *cache) { delete cache; }

int ds_moe_cache_record(ds_moe_cache *cache, int32_t layer, const int32_t *counts, int32_t *fills,
                        int32_t *n_fills) {
  if (!cache || !counts || layer < 0 || layer >= cache->n_layers) return DS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(cache->mu);
  std::vector<int32_t> f;
  std::vector<char> changed((size_t)cache->n_layers, 0);
  cache->record(layer, counts, f, changed);
  if (fills) memcpy(fills, f.data(), sizeof(int32_t) * f.size());
  if (n_fills) *n_fills = (int32_t)(f.size() / 2);
  return DS_OK;
}

int ds_moe_cache_slot(const ds_moe_cache *cache, int32_t layer, int32_t expert, int32_t *slot) {
  if (!cache || !slot || layer < 0 || layer >= cache->n_layers || expert < 0 || expert >= cache->E)
    return DS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(cache->mu);
  *slot = cache->table[(size_t)layer * cache->E + expert];
  return DS_OK;
}

int ds_moe_cache_stats(const ds_moe_cache *cache, int64_t *hits, int64_t *misses, int64_t *resident) {
  if (!cache) return DS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(cache->mu);
  if (hits) *hits = cache->hits;
  if (misses) *misses = cache->misses;
  if (resident) {
    int64_t n = 0;
    for (int32_t o : cache->owner_e) n += o >= 0;
    *resident = n;
  }
  return DS_OK;
}

int ds_moe_cache_layer(ds_moe_cache *cache, int32_t layer, const ds_moe_weights *weights, const void *x, int64_t T,
                       float *out, void *workspace, size_t workspace_bytes, void *stream, char *err,
                       size_t errlen) {
  if (!cache || layer < 0 || layer >= cache->n_layers)
    return cfail(err, errlen, DS_ERR_INVALID_ARG, "bad cache or layer");
  if (!cache->tables) return cfail(err, errlen, DS_ERR_INVALID_ARG, "the cache was created without device tables");
  ds_moe_shape shape{cache->sh.D, cache->sh.E, cache->sh.F, cache->sh.Fs, cache->sh.k, cache->sh.x_dtype,
                     cache->sh.router_dtype, cache->sh.routed_scale, cache->sh.logit_scale,
                     cache->sh.bias_select_only, cache->sh.fmt};
  ds_moe_residency res{cache->tables + (size_t)layer * cache->E, cache->slots, cache->host[layer]};
  int rc = ds_moe_layer_resident(&shape, weights, &res, x, T, out, workspace, workspace_bytes, nullptr, stream, err,
                                 errlen);
  if (rc || T == 0) return rc;
  // the experts this call used, then the fills for later calls (same stream)
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<int32_t> counts((size_t)cache->E);
  cudaError_t e = cudaMemcpyAsync(counts.data(), dsm::workspace_counts(cache->sh, T, workspace),
                                  sizeof(int32_t) * cache->E, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cfail(err, errlen, DS_ERR_CUDA, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(cache->mu);
  std::vector<int32_t> fills;
  std::vector<char> changed((size_t)cache->n_layers, 0);
  cache->record(layer, counts.data(), fills, changed);
  for (size_t i = 0; i < fills.size(); i += 2) {
    const int64_t slot = fills[i], ex = fills[i + 1];
    e = cudaMemcpyAsync(cache->slots + slot * cache->eb, cache->host[layer] + ex * cache->eb, (size_t)cache->eb,
                        cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cfail(err, errlen, DS_ERR_CUDA, cudaGetErrorString(e));
  }
  for (int32_t l = 0; l < cache->n_layers; ++l)
    if (changed[l]) {
      // pageable source: staged before the call returns, ordered on the stream
      e = cudaMemcpyAsync(cache->tables + (size_t)l * cache->E, cache->table.data() + (size_t)l * cache->E,
                          sizeof(int32_t) * cache->E, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cfail(err, errlen, DS_ERR_CUDA, cudaGetErrorString(e));
    }
  return DS_OK;
}

}  // extern "C"
