/* ds_moe: one routed mixture-of-experts layer with 2-bit (Q2_K) or 4-bit
 * (Q4_K) routed experts, computed on one GB300 (sm_103a) GPU.
 *
 * The layer ("Understanding Dwarf Star", 5.3.2 "The MoE Architecture" and
 * 5.3.7 "The MoE Kernel in Metal"):
 *     logits  = x W_router^T (+ bias)                      router, fp32
 *     ids, w  = top-k of logits, w = softmax over the k     selection
 *     y_e(x)  = W_down,e ( SiLU(W_gate,e x) * (W_up,e x) )  SwiGLU expert
 *     out     = y_shared(x) + sum_j w_j y_{ids_j}(x)        combine, fp32
 * with the routed expert matrices stored as Q2_K super-blocks ("Understanding
 * Dwarf Star", 3.3.3 "Q2_K: 2.625 Bits Per Element"): 84 bytes per 256
 * weights along each matrix's input dimension (or Q4_K, below).  Shapes of the DeepSeek V4
 * Flash layer: n_embd 4096, 256 experts, top-6, one shared expert, expert
 * width 2048 ("Understanding Dwarf Star", 2.4.3 shape table).
 *
 * Conventions (the pages' C engine style: int status, 0 = ok, negative =
 * error, plus a caller-supplied error buffer; caller-owned scratch):
 *   - Every pointer is a DEVICE pointer unless the argument says "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream unless stated.
 *   - The library allocates no device memory for a call: the caller owns
 *     every buffer, including the workspace, and nothing is retained after a
 *     call returns.  (Per device it keeps one status word, and
 *     ds_moe_layer_noalloc's static scratch; ds_moe_cache keeps host state.)
 *   - Argument errors are detected on the host before any launch and return
 *     DS_ERR_INVALID_ARG (or DS_ERR_UNSUPPORTED) with a message in err.
 *     Errors a kernel detects (a non-finite weight given to the quantiser,
 *     a corrupted id, a timed-out wait) are recorded in a per-device sticky
 *     status word, read and cleared by ds_moe_sync_status.
 *   - err may be NULL; otherwise up to errlen bytes (NUL-terminated) are
 *     written on failure.
 *   - Calls are thread-safe as long as concurrent calls use distinct
 *     workspaces and outputs.
 *
 * Q2_K super-block (84 bytes, 256 weights):
 *   bytes [0,16)   sub-block s (16 weights each): scale sc_s in the low
 *                  nibble, min m_s in the high nibble
 *   bytes [16,80)  2-bit codes; weight j at byte 16 + j/4, bits 2*(j%4)
 *   bytes [80,82)  d, fp16 little-endian;  bytes [82,84) dmin, fp16
 *   weight j = d*sc_s*q_j - dmin*m_s  (s = j/16)
 * Q4_K super-block (144 bytes, 256 weights; "Understanding Dwarf Star",
 * 2.3.2 "K-Quant Formats": d at 0, dmin at 2, 12 bytes of 6-bit scales and
 * mins at 4, 128 bytes of 4-bit codes at 16, 8 sub-blocks of 32):
 *   bytes [0,2) d, [2,4) dmin, fp16 little-endian
 *   bytes [4,16)   one 96-bit little-endian integer: field i in bits
 *                  [6i, 6i+6); fields 0..7 = sc_s, 8..15 = m_s
 *   bytes [16,144) 4-bit codes; weight j at byte 16 + j/2, low nibble for
 *                  even j
 *   weight j = d*sc_s*q_j - dmin*m_s  (s = j/32)
 * A row of in_dim weights uses ceil(in_dim/256) blocks (zero-padded).
 * Packed expert e = gate [n_ff rows][n_embd] | up [n_ff][n_embd] |
 * down [n_embd rows][n_ff], each row-major in blocks; experts are contiguous
 * in expert order, each ds_moe_expert_bytes_fmt() long; base 16-byte aligned.
 */
#ifndef DS_MOE_H
#define DS_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = -1,  /* bad pointer, size, alignment or workspace    */
  DS_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. odd n_embd)  */
  DS_ERR_CUDA = -3,         /* a CUDA runtime call failed                    */
  DS_ERR_TIMEOUT = -4,      /* a device wait hit its iteration limit         */
  DS_ERR_DEVICE_CHECK = -5  /* a kernel found invalid data                   */
} ds_status;

typedef enum { DS_F32 = 0, DS_BF16 = 1 } ds_dtype;

/* Storage format of the routed experts. */
typedef enum { DS_Q2_K = 0, DS_Q4_K = 1 } ds_expert_format;

typedef struct {
  int32_t n_embd;       /* D: model width, multiple of 256, <= 8192          */
  int32_t n_expert;     /* E: routed experts, 1..1024                        */
  int32_t n_ff;         /* F: expert width, multiple of 128, <= 8192         */
  int32_t n_ff_shared;  /* Fs: shared expert width, 0 = none, mult. of 128, <= 8192 */
  int32_t top_k;        /* k: 1..min(E, 16)                                  */
  int32_t x_dtype;      /* ds_dtype of x                                     */
  int32_t router_dtype; /* ds_dtype of router_w                              */
  float routed_scale;   /* multiplies the k routing weights (1.0 default)    */
  float logit_scale;    /* multiplies the selected logits before their softmax
                           (the other reading of [UDS] 5.3.5's 1.5 "before
                           softmax"); 1 = plain softmax, 0 is taken as 1; the
                           selection does not depend on it                  */
  int32_t bias_select_only; /* 0: router_bias is part of the logits (selection
                           and weights); 1: it steers the selection only and
                           the weights use the logits without it            */
  int32_t expert_format; /* ds_expert_format of the routed experts (0 = Q2_K) */
} ds_moe_shape;

typedef struct {
  const void *router_w;       /* [E][D] router_dtype, row-major                 */
  const float *router_bias;   /* [E] fp32 added to the logits, or NULL          */
  const uint16_t *shared_gate; /* [Fs][D] bf16 bits (NULL when Fs == 0)        */
  const uint16_t *shared_up;   /* [Fs][D] bf16 bits                             */
  const uint16_t *shared_down; /* [D][Fs] bf16 bits                             */
  const uint8_t *experts;    /* [E] packed experts in expert_format, 16-byte aligned */
} ds_moe_weights;

/* Optional debug outputs of ds_moe_layer (device pointers; NULL fields and a
 * NULL struct are skipped).  All are written in the same stream order. */
typedef struct {
  float *logits;    /* [T][E] router logits incl. bias (fp32)                 */
  int32_t *ids;     /* [T][k] selected experts, descending logit order        */
  float *w;         /* [T][k] routing weights (after routed_scale)            */
  int32_t *counts;  /* [E] tokens per expert                                  */
  int32_t *offsets; /* [E+1] exclusive scan of counts                         */
  int32_t *perm;    /* [T*k] pair t*k+j at position offsets[e]+rank, stable   */
} ds_moe_debug;

/* Bytes of a Q2_K matrix of `rows` rows of `in_dim` weights:
 * rows * ceil(in_dim/256) * 84 ("Understanding Dwarf Star", 3.3.3).
 * Returns 0 for negative sizes. */
size_t ds_moe_q2k_bytes(int64_t rows, int64_t in_dim);

/* Bytes of a Q4_K matrix: rows * ceil(in_dim/256) * 144 ("Understanding
 * Dwarf Star", 2.3.2).  Returns 0 for negative sizes. */
size_t ds_moe_q4k_bytes(int64_t rows, int64_t in_dim);

/* Bytes of one packed routed expert (gate, up and down; "The sparsity that
 * pays for everything else in DwarfStar", "Where the parameters actually
 * are": gate, up and down per expert), Q2_K. */
size_t ds_moe_expert_bytes(int32_t n_embd, int32_t n_ff);

/* The same in a given ds_expert_format; 0 for an unknown format. */
size_t ds_moe_expert_bytes_fmt(int32_t expert_format, int32_t n_embd, int32_t n_ff);

/* Quantise an fp32 matrix w [rows][in_dim] (row-major, device) to Q2_K
 * blocks in out (ds_moe_q2k_bytes(rows, in_dim) bytes, device, 4-byte
 * aligned).  The encoding picks, per super-block, the smallest fp16 dmin and
 * d and the smallest 4-bit mins and scales whose four evenly spaced levels
 * cover each 16-weight sub-block, then rounds each weight to its nearest
 * level, ties upward ("Understanding Dwarf Star", 2.3.5: Q2_K levels are
 * evenly spaced between the block's min and max; 3.3.3 block layout).  Every
 * decision is exact, so the bytes are a pure function of the inputs.
 * Non-finite inputs or |w| > 65504 set DS_ERR_DEVICE_CHECK in the status
 * word and produce an all-zero block. */
int ds_moe_quantize_q2k(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, void *stream,
                        char *err, size_t errlen);

/* Dequantise Q2_K blocks q [rows][ceil(in_dim/256)*84] to fp32
 * out [rows][in_dim]: out = fp32(d*sc*q - dmin*m), i.e. the exact value
 * rounded once ("Understanding Dwarf Star", 2.8.1: weights are rebuilt from
 * the stored scales and mins).  A test and inspection aid. */
int ds_moe_dequantize_q2k(const uint8_t *q, int64_t rows, int64_t in_dim, float *out, void *stream,
                          char *err, size_t errlen);

/* Quantise to Q4_K blocks (ds_moe_q4k_bytes(rows, in_dim) bytes, device,
 * 4-byte aligned).  The same search as for Q2_K with 4-bit codes and 6-bit
 * scales and mins, per 32-weight sub-block: the smallest fp16 dmin with
 * 63*dmin >= max(-min), the smallest m_s <= 63 covering each sub-block's
 * minimum, the smallest fp16 d with 945*d >= max(hi_s + b_s), the smallest
 * sc_s <= 63 with 15*d*sc_s >= hi_s + b_s, then the nearest of the 16 levels,
 * ties upward ("Understanding Dwarf Star", 2.3.2 layout; 2.3.5 evenly spaced
 * levels).  Exact, like the Q2_K quantiser; the same input checks. */
int ds_moe_quantize_q4k(const float *w, int64_t rows, int64_t in_dim, uint8_t *out, void *stream,
                        char *err, size_t errlen);

/* Dequantise Q4_K blocks to fp32: fp32(d*sc*q - dmin*m), rounded once. */
int ds_moe_dequantize_q4k(const uint8_t *q, int64_t rows, int64_t in_dim, float *out, void *stream,
                          char *err, size_t errlen);

/* Workspace bytes ds_moe_layer needs for T tokens of this shape (host call,
 * synchronous).  The workspace must be 256-byte aligned. */
int ds_moe_workspace_bytes(const ds_moe_shape *shape, int64_t T, size_t *bytes, char *err,
                           size_t errlen);

/* One routed MoE layer on T tokens (the equations at the top of this file).
 *   x    [T][D] x_dtype (device), 16-byte aligned
 *   out  [T][D] fp32 (device), 16-byte aligned; fully overwritten
 *   workspace: ds_moe_workspace_bytes bytes, 256-byte aligned, caller-owned;
 *        its contents need no initialisation and are scratch after return
 *   dbg  optional debug outputs (NULL to skip)
 * Tokens are independent: row t of out depends only on row t of x.
 * A NaN router logit is never selected.  When fewer than top_k of a token's
 * logits are numbers (a NaN in its x, say), its remaining picks take expert
 * 0, its row of out is not meaningful, and ds_moe_sync_status reports
 * DS_ERR_DEVICE_CHECK; nothing of such a call carries over into later calls.
 * T == 0 is a no-op.  The kernels that run depend on T and the shape (see
 * ds_moe_layer_path): one token at the instantiated widths with top_k <= 8
 * streams the whole layer through one cooperative kernel; up to four tokens
 * (and one token otherwise) use a three-kernel decode chain, except where
 * the batched kernels below apply; both compute the routed rows as exact
 * integer dots on 16-bit fixed-point activations.  4..16 tokens with Q2_K
 * experts, bf16 x and router and n_embd, n_ff, n_ff_shared multiples of
 * 1024 run the batched decode kernels (the same integer dots; the shared
 * expert on the tensor cores with exact bf16 products).  Larger batches with bf16 x and router and n_embd, n_ff
 * multiples of 1024 (Q4_K experts: from five tokens) run the expert FFNs as
 * grouped tcgen05 GEMMs with fp16 operands (dequantised weights and
 * activations rounded once to fp16; an |x| or intermediate above 65504 is
 * saturated and reported by ds_moe_sync_status as DS_ERR_DEVICE_CHECK);
 * every other case uses the grouped dequantising GEMV path with fp32
 * arithmetic. */
int ds_moe_layer(const ds_moe_shape *shape, const ds_moe_weights *weights, const void *x, int64_t T,
                 float *out, void *workspace, size_t workspace_bytes, const ds_moe_debug *dbg,
                 void *stream, char *err, size_t errlen);

/* ds_moe_layer with x and out in HOST memory (pinned for best speed): the
 * host-to-device copy of x and the device-to-host copy of out are issued on
 * `stream` around the layer, using the workspace for the device copies
 * (ds_moe_workspace_bytes covers them).  When the one-token kernel serves
 * the call (T == 1 at its widths) and the device can address both buffers
 * (pinned memory), no copy operation is issued: the router grid reads x in
 * host memory and keeps a device copy in the workspace for the streaming
 * kernel, which writes out straight into host memory.  Returns after
 * enqueueing; the caller synchronises the stream before reading out. */
int ds_moe_layer_hostio(const ds_moe_shape *shape, const ds_moe_weights *weights,
                        const void *x_host, int64_t T, float *out_host, void *workspace,
                        size_t workspace_bytes, void *stream, char *err, size_t errlen);

/* A stack of n_layers blocks, each  x <- x + layer_l(bf16(RMSNorm(x)))  with
 * RMSNorm(x) = x / sqrt(mean(x^2) + eps) and unit gain (pages: every layer
 * applies RMSNorm and a residual connection).  x [T][D] fp32 (device) is the
 * residual stream, updated in place.  layers: host array of n_layers weight
 * sets; shape->x_dtype must be DS_BF16.  Workspace as for ds_moe_layer. */
int ds_moe_stack(const ds_moe_shape *shape, const ds_moe_weights *layers, int32_t n_layers,
                 float *x, int64_t T, float eps, void *workspace, size_t workspace_bytes,
                 void *stream, char *err, size_t errlen);

/* ds_moe_stack with a format per layer ("q2-q4" mixed stacks: most layers
 * Q2_K, the last few Q4_K).  formats: host array of n_layers
 * ds_expert_format values that replace shape->expert_format for each layer,
 * or NULL (every layer as the shape says).  The workspace must hold
 * ds_moe_workspace_bytes of the shape with expert_format = DS_Q2_K when any
 * layer is Q2_K, else with DS_Q4_K.  A bad format entry returns
 * DS_ERR_INVALID_ARG before any launch. */
int ds_moe_stack_mixed(const ds_moe_shape *shape, const ds_moe_weights *layers,
                       const int32_t *formats, int32_t n_layers, float *x, int64_t T, float eps,
                       void *workspace, size_t workspace_bytes, void *stream, char *err,
                       size_t errlen);

/* ds_moe_layer for callers that cannot allocate device memory where they
 * call the layer: a plugin or extension inside a host program whose own
 * allocator owns all device memory, or a real-time loop that must not take
 * cudaMalloc's implicit device-wide synchronisation.  It takes no workspace:
 * its scratch is a static 64 MiB device array inside this library, allocated
 * on each GPU when the library is loaded there and held until the process
 * exits.  The pages have no counterpart to this entry point.
 *   x, T, out, stream, err: as for ds_moe_layer (no debug outputs); the
 *   arguments are validated in the same order, so T == 0 with bad weights
 *   is rejected as ds_moe_layer rejects it.
 *   Rejects, with DS_ERR_INVALID_ARG and a message, any T whose
 *   ds_moe_workspace_bytes exceeds 64 MiB (at the 4096/256/6/2048 shape the
 *   limit is reached at about 200 tokens; from 17 tokens the tensor-core
 *   path's scratch includes a 16.8 MB fp16 copy of the shared down matrix).
 *   Allocates nothing: no cudaMalloc, no cudaFree.
 *   The first call on a device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 *   Every call reuses the same array and leaves its contents behind; the
 *   call clears what must start at zero.  Calls that overlap on the GPU
 *   (other streams or threads) race on the array: serialise them. */
int ds_moe_layer_noalloc(const ds_moe_shape *shape, const ds_moe_weights *weights, const void *x,
                         int64_t T, float *out, void *stream, char *err, size_t errlen);

/* Expert residency beyond device memory ("The sparsity that pays for
 * everything else in DwarfStar", "Page the experts off the SSD" and "The
 * cache is never allowed to become a correctness structure": routed experts
 * are paged in through a cache, and the output does not depend on what the
 * cache holds).  Here every routed expert of a layer has a copy in host
 * memory the device can address (pinned and mapped by cudaHostAlloc,
 * registered by cudaHostRegister, or the memory of a coherent host such as
 * Grace, read over NVLink-C2C), and a caller-owned pool of device slots holds
 * some of them.
 *   slot          [E] int32 (device): the cache slot of expert e, or -1
 *   cache         device: slots of ds_moe_expert_bytes_fmt() bytes each,
 *                 16-byte aligned (may be NULL when no slot is in use)
 *   experts_host  HOST pointer to the layer's E packed experts (the layout of
 *                 ds_moe_weights.experts), 16-byte aligned */
typedef struct {
  const int32_t *slot;
  const uint8_t *cache;
  const uint8_t *experts_host;
} ds_moe_residency;

/* ds_moe_layer with the routed experts read through a residency view: each
 * expert from its cache slot, or from the host copy (ordinary loads) when it
 * has none; weights->experts is ignored and may be NULL.  The same kernels
 * run on the same bytes wherever an expert lives, so the output is
 * bit-identical for every slot table.  Kernels: as ds_moe_layer for up to
 * four tokens at the instantiated widths (the streaming kernel, the
 * three-kernel chain), the grouped dequantising GEMV path otherwise
 * (ds_moe_layer_path_resident).  Errors as ds_moe_layer, and
 * DS_ERR_INVALID_ARG for a missing slot table or a host copy the device
 * cannot address. */
int ds_moe_layer_resident(const ds_moe_shape *shape, const ds_moe_weights *weights,
                          const ds_moe_residency *residency, const void *x, int64_t T, float *out,
                          void *workspace, size_t workspace_bytes, const ds_moe_debug *dbg, void *stream,
                          char *err, size_t errlen);

/* A cache of routed experts for n_layers layers of one shape (opaque host
 * object).  experts_host: host array of n_layers host pointers, each a
 * layer's E packed experts in device-addressable host memory (as for
 * ds_moe_residency).  slots: caller-owned device buffer of n_slots experts
 * (ds_moe_expert_bytes_fmt() bytes each, 16-byte aligned; the byte budget of
 * the cache); tables: caller-owned device buffer of n_layers * E int32 slot
 * tables, set here (synchronously) to "every expert in host memory".  With
 * tables == NULL the object only plans (ds_moe_cache_record; no device
 * memory is touched).  The library allocates no device memory; the object
 * itself is host memory, freed by ds_moe_cache_destroy. */
typedef struct ds_moe_cache ds_moe_cache;
int ds_moe_cache_create(const ds_moe_shape *shape, int32_t n_layers, const void *const *experts_host,
                        void *slots, int64_t n_slots, int32_t *tables, ds_moe_cache **cache, char *err,
                        size_t errlen);
void ds_moe_cache_destroy(ds_moe_cache *cache);

/* One layer through the cache: ds_moe_layer_resident with this layer's slot
 * table, then (after synchronising the stream to read which experts the call
 * used) the experts it missed are copied on `stream` into free slots or the
 * least recently used slots that this call did not use, and the slot tables
 * are updated on `stream` for the calls that follow.  The output does not
 * depend on the cache's contents.  Not for use inside stream capture (it
 * synchronises the stream). */
int ds_moe_cache_layer(ds_moe_cache *cache, int32_t layer, const ds_moe_weights *weights, const void *x, int64_t T,
                       float *out, void *workspace, size_t workspace_bytes, void *stream, char *err,
                       size_t errlen);

/* The cache policy alone, on the host: record that a call of `layer` used
 * the experts with counts[e] > 0 (host array [E]).  Hits refresh their
 * slots; each miss takes a free slot, else the least recently used slot not
 * used by this call (none: the expert stays in host memory).  fills (host,
 * optional, 2 * E int32) receives (slot, expert) pairs of the copies to make,
 * n_fills their number.  ds_moe_cache_layer does this after every call. */
int ds_moe_cache_record(ds_moe_cache *cache, int32_t layer, const int32_t *counts, int32_t *fills,
                        int32_t *n_fills);
/* *slot = the slot of expert `expert` of `layer` (host mirror of the
 * tables), or -1 when it is in host memory.  DS_ERR_INVALID_ARG for a bad
 * cache, layer, expert or NULL slot. */
int ds_moe_cache_slot(const ds_moe_cache *cache, int32_t layer, int32_t expert, int32_t *slot);
/* Counters since creation: experts found in a slot, experts read from host
 * memory, and slots in use. */
int ds_moe_cache_stats(const ds_moe_cache *cache, int64_t *hits, int64_t *misses, int64_t *resident);

/* Which kernels ds_moe_layer runs for T tokens of this shape with this x
 * pointer (host call; nothing is launched).  Returns one of the DS_PATH_*
 * values, or DS_ERR_INVALID_ARG for a shape ds_moe_layer would reject. */
enum {
  DS_PATH_NONE = 0,          /* T == 0 */
  DS_PATH_STREAM = 1,        /* one token: router kernel + one cooperative streaming kernel */
  DS_PATH_DECODE3 = 2,       /* T <= 4 (2..3, or 4 where the batched kernels do not apply): router,
                                gate/up and down kernels chained */
  DS_PATH_GROUPED_GEMV = 3,  /* route kernels + grouped dequantising GEMVs + combine */
  DS_PATH_TENSOR_CORE = 4,   /* route kernels + grouped tcgen05 GEMMs + combine */
  DS_PATH_BATCHED_DECODE = 5 /* 4..16 tokens: router kernel + batched decode kernels (integer
                                routed dots, shared expert on the tensor cores) */
};
int ds_moe_layer_path(const ds_moe_shape *shape, int64_t T, const void *x);
/* The same for ds_moe_layer_resident. */
int ds_moe_layer_path_resident(const ds_moe_shape *shape, int64_t T);

/* Synchronise `stream`, then read and clear this device's sticky status
 * word (one atomic exchange on the device, so bits that kernels on other
 * streams set meanwhile are not lost: they are reported by the next call).
 * Returns DS_OK, DS_ERR_TIMEOUT or DS_ERR_DEVICE_CHECK (with a message
 * naming the check), or DS_ERR_CUDA if the stream itself failed. */
int ds_moe_sync_status(void *stream, char *err, size_t errlen);

/* Library version string (static storage). */
const char *ds_moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_MOE_H */
