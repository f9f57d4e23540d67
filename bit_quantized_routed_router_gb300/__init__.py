"""Python binding of the ds_moe C ABI (``include/ds_moe.h``).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``libds_moe.so``.  PyTorch supplies device memory and streams.  There is
no fallback: if the library has not been built, importing the binding's
functions raises.

Names mirror the C entry points: ``q2k_bytes``, ``expert_bytes``,
``quantize_q2k``, ``dequantize_q2k``, ``workspace_bytes``, ``layer``,
``layer_hostio``, ``stack``, ``sync_status``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libds_moe.so")

DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED = 0, -1, -2
DS_ERR_CUDA, DS_ERR_TIMEOUT, DS_ERR_DEVICE_CHECK = -3, -4, -5
DS_F32, DS_BF16 = 0, 1
DS_Q2_K, DS_Q4_K = 0, 1

SYMBOLS = ["ds_moe_q2k_bytes", "ds_moe_expert_bytes", "ds_moe_quantize_q2k",
           "ds_moe_dequantize_q2k", "ds_moe_workspace_bytes", "ds_moe_layer",
           "ds_moe_layer_hostio", "ds_moe_stack", "ds_moe_sync_status", "ds_moe_version",
           "ds_moe_layer_noalloc", "ds_moe_layer_path", "ds_moe_q4k_bytes",
           "ds_moe_expert_bytes_fmt", "ds_moe_quantize_q4k", "ds_moe_dequantize_q4k",
           "ds_moe_stack_mixed", "ds_moe_layer_resident", "ds_moe_layer_path_resident",
           "ds_moe_cache_create", "ds_moe_cache_destroy", "ds_moe_cache_layer", "ds_moe_cache_record",
           "ds_moe_cache_slot", "ds_moe_cache_stats"]

# ds_moe_layer_path results
PATH_NONE, PATH_STREAM, PATH_DECODE3, PATH_GROUPED_GEMV, PATH_TENSOR_CORE, PATH_BATCHED_DECODE = 0, 1, 2, 3, 4, 5


class DsMoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"ds_moe error {code}: {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("n_embd", ctypes.c_int32), ("n_expert", ctypes.c_int32),
                ("n_ff", ctypes.c_int32), ("n_ff_shared", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("x_dtype", ctypes.c_int32),
                ("router_dtype", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("logit_scale", ctypes.c_float), ("bias_select_only", ctypes.c_int32),
                ("expert_format", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("shared_gate", ctypes.c_void_p), ("shared_up", ctypes.c_void_p),
                ("shared_down", ctypes.c_void_p), ("experts", ctypes.c_void_p)]


class Residency(ctypes.Structure):
    _fields_ = [("slot", ctypes.c_void_p), ("cache", ctypes.c_void_p), ("experts_host", ctypes.c_void_p)]


class Debug(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libds_moe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                               "(or python bit_quantized_routed_router_gb300/build.py)")
        _lib = load(LIB_PATH)
    return _lib


def load(path: str):
    """A build of the library at `path` (ctypes handle with its signatures)."""
    L = ctypes.CDLL(path)
    vp, i64, sz, cp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_char_p
    L.ds_moe_q2k_bytes.restype = sz
    L.ds_moe_q2k_bytes.argtypes = [i64, i64]
    L.ds_moe_q4k_bytes.restype = sz
    L.ds_moe_q4k_bytes.argtypes = [i64, i64]
    L.ds_moe_expert_bytes.restype = sz
    L.ds_moe_expert_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.ds_moe_expert_bytes_fmt.restype = sz
    L.ds_moe_expert_bytes_fmt.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    for f in (L.ds_moe_quantize_q2k, L.ds_moe_dequantize_q2k, L.ds_moe_quantize_q4k,
              L.ds_moe_dequantize_q4k):
        f.restype = ctypes.c_int
        f.argtypes = [vp, i64, i64, vp, vp, cp, sz]
    L.ds_moe_workspace_bytes.restype = ctypes.c_int
    L.ds_moe_workspace_bytes.argtypes = [ctypes.POINTER(Shape), i64, ctypes.POINTER(sz), cp, sz]
    L.ds_moe_layer.restype = ctypes.c_int
    L.ds_moe_layer.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), vp, i64, vp, vp,
                               sz, ctypes.POINTER(Debug), vp, cp, sz]
    L.ds_moe_layer_hostio.restype = ctypes.c_int
    L.ds_moe_layer_hostio.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), vp, i64,
                                      vp, vp, sz, vp, cp, sz]
    L.ds_moe_stack.restype = ctypes.c_int
    L.ds_moe_stack.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), ctypes.c_int32,
                               vp, i64, ctypes.c_float, vp, sz, vp, cp, sz]
    L.ds_moe_stack_mixed.restype = ctypes.c_int
    L.ds_moe_stack_mixed.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), vp,
                                     ctypes.c_int32, vp, i64, ctypes.c_float, vp, sz, vp, cp, sz]
    L.ds_moe_layer_noalloc.restype = ctypes.c_int
    L.ds_moe_layer_noalloc.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), vp, i64,
                                       vp, vp, cp, sz]
    L.ds_moe_sync_status.restype = ctypes.c_int
    L.ds_moe_sync_status.argtypes = [vp, cp, sz]
    L.ds_moe_version.restype = ctypes.c_char_p
    L.ds_moe_version.argtypes = []
    L.ds_moe_layer_resident.restype = ctypes.c_int
    L.ds_moe_layer_resident.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights),
                                        ctypes.POINTER(Residency), vp, i64, vp, vp, sz,
                                        ctypes.POINTER(Debug), vp, cp, sz]
    L.ds_moe_layer_path_resident.restype = ctypes.c_int
    L.ds_moe_layer_path_resident.argtypes = [ctypes.POINTER(Shape), i64]
    L.ds_moe_cache_create.restype = ctypes.c_int
    L.ds_moe_cache_create.argtypes = [ctypes.POINTER(Shape), ctypes.c_int32, ctypes.POINTER(vp), vp, i64,
                                      vp, ctypes.POINTER(vp), cp, sz]
    L.ds_moe_cache_destroy.restype = None
    L.ds_moe_cache_destroy.argtypes = [vp]
    L.ds_moe_cache_layer.restype = ctypes.c_int
    L.ds_moe_cache_layer.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(Weights), vp, i64, vp, vp, sz, vp,
                                     cp, sz]
    L.ds_moe_cache_record.restype = ctypes.c_int
    L.ds_moe_cache_record.argtypes = [vp, ctypes.c_int32, vp, vp, ctypes.POINTER(ctypes.c_int32)]
    L.ds_moe_cache_slot.restype = ctypes.c_int
    L.ds_moe_cache_slot.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    L.ds_moe_cache_stats.restype = ctypes.c_int
    L.ds_moe_cache_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
    return L


def _call(fn, *args):
    err = ctypes.create_string_buffer(512)
    rc = fn(*args, err, 512)
    if rc != DS_OK:
        raise DsMoeError(rc, err.value.decode(errors="replace"))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


@dataclass
class MoEShape:
    n_embd: int
    n_expert: int
    n_ff: int
    n_ff_shared: int
    top_k: int
    x_dtype: int = DS_BF16
    router_dtype: int = DS_BF16
    routed_scale: float = 1.0
    logit_scale: float = 1.0
    bias_select_only: int = 0
    expert_format: int = 0  # DS_Q2_K or DS_Q4_K

    def c(self) -> Shape:
        return Shape(self.n_embd, self.n_expert, self.n_ff, self.n_ff_shared, self.top_k,
                     self.x_dtype, self.router_dtype, self.routed_scale, self.logit_scale,
                     self.bias_select_only, self.expert_format)


@dataclass
class MoEWeights:
    """Device tensors of one layer (see include/ds_moe.h for layouts)."""
    router_w: object
    experts: object
    router_bias: object = None
    shared_gate: object = None
    shared_up: object = None
    shared_down: object = None

    def c(self) -> Weights:
        return Weights(_ptr(self.router_w), _ptr(self.router_bias), _ptr(self.shared_gate),
                       _ptr(self.shared_up), _ptr(self.shared_down), _ptr(self.experts))


def version() -> str:
    return lib().ds_moe_version().decode()


def q2k_bytes(rows: int, in_dim: int) -> int:
    return lib().ds_moe_q2k_bytes(rows, in_dim)


def q4k_bytes(rows: int, in_dim: int) -> int:
    return lib().ds_moe_q4k_bytes(rows, in_dim)


def expert_bytes(n_embd: int, n_ff: int, expert_format: int = 0) -> int:
    return lib().ds_moe_expert_bytes_fmt(expert_format, n_embd, n_ff)


def quantize_q2k(w, out, stream=None):
    """w: fp32 device tensor [rows][in_dim]; out: uint8 device tensor of q2k_bytes."""
    rows, in_dim = w.shape
    _call(lib().ds_moe_quantize_q2k, w.data_ptr(), rows, in_dim, out.data_ptr(), _stream(stream))


def dequantize_q2k(q, rows, in_dim, out, stream=None):
    _call(lib().ds_moe_dequantize_q2k, q.data_ptr(), rows, in_dim, out.data_ptr(), _stream(stream))


def quantize_q4k(w, out, stream=None):
    """w: fp32 device tensor [rows][in_dim]; out: uint8 device tensor of q4k_bytes."""
    rows, in_dim = w.shape
    _call(lib().ds_moe_quantize_q4k, w.data_ptr(), rows, in_dim, out.data_ptr(), _stream(stream))


def dequantize_q4k(q, rows, in_dim, out, stream=None):
    _call(lib().ds_moe_dequantize_q4k, q.data_ptr(), rows, in_dim, out.data_ptr(), _stream(stream))


def layer_path(shape: MoEShape, T: int, x=None) -> int:
    """Which kernels ds_moe_layer runs for T tokens (a PATH_* value)."""
    L = lib()
    L.ds_moe_layer_path.restype = ctypes.c_int
    L.ds_moe_layer_path.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    sh = shape.c()
    rc = L.ds_moe_layer_path(ctypes.byref(sh), T, _ptr(x) if x is not None else 256)
    if rc < 0:
        raise DsMoeError(rc, "shape rejected")
    return rc


def workspace_bytes(shape: MoEShape, T: int) -> int:
    n = ctypes.c_size_t(0)
    _call(lib().ds_moe_workspace_bytes, ctypes.byref(shape.c()), T, ctypes.byref(n))
    return n.value


def layer(shape: MoEShape, weights: MoEWeights, x, out, workspace, debug: dict | None = None,
          stream=None, T: int | None = None):
    """out[T][D] fp32 = MoE layer of x[T][D] (device tensors)."""
    T = x.shape[0] if T is None else T
    dbg = None
    if debug is not None:
        dbg = ctypes.byref(Debug(*[_ptr(debug.get(n)) for n in
                                   ("logits", "ids", "w", "counts", "offsets", "perm")]))
    _call(lib().ds_moe_layer, ctypes.byref(shape.c()), ctypes.byref(weights.c()), x.data_ptr(), T,
          out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), dbg,
          _stream(stream))


def layer_hostio(shape: MoEShape, weights: MoEWeights, x_host, out_host, workspace, stream=None):
    """Same as layer with x and out in (pinned) host memory; enqueues only."""
    _call(lib().ds_moe_layer_hostio, ctypes.byref(shape.c()), ctypes.byref(weights.c()),
          x_host.data_ptr(), x_host.shape[0], out_host.data_ptr(), workspace.data_ptr(),
          workspace.numel() * workspace.element_size(), _stream(stream))


def layer_noalloc(shape: MoEShape, weights: MoEWeights, x, out, stream=None, T: int | None = None):
    """layer() without a workspace: the library's static device scratch is used
    (for callers that cannot allocate; at most 64 MiB of scratch, serialise calls)."""
    T = x.shape[0] if T is None else T
    _call(lib().ds_moe_layer_noalloc, ctypes.byref(shape.c()), ctypes.byref(weights.c()),
          x.data_ptr(), T, out.data_ptr(), _stream(stream))


def layer_resident(shape: MoEShape, weights: MoEWeights, slot, cache, experts_host, x, out, workspace,
                   debug: dict | None = None, stream=None, T: int | None = None):
    """layer() with the routed experts read through a residency view: slot [E]
    int32 (device, -1 = host), cache (device slots or None), experts_host (a
    pinned host tensor of the E packed experts)."""
    T = x.shape[0] if T is None else T
    dbg = None
    if debug is not None:
        dbg = ctypes.byref(Debug(*[_ptr(debug.get(n)) for n in
                                   ("logits", "ids", "w", "counts", "offsets", "perm")]))
    res = Residency(_ptr(slot), _ptr(cache), _ptr(experts_host))
    _call(lib().ds_moe_layer_resident, ctypes.byref(shape.c()), ctypes.byref(weights.c()), ctypes.byref(res),
          x.data_ptr(), T, out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
          dbg, _stream(stream))


def layer_path_resident(shape: MoEShape, T: int) -> int:
    rc = lib().ds_moe_layer_path_resident(ctypes.byref(shape.c()), T)
    if rc < 0:
        raise DsMoeError(rc, "invalid shape or T")
    return rc


class ExpertCache:
    """A cache of routed experts in device slots for n_layers layers (the C
    object ds_moe_cache).  experts_host: per layer a pinned host tensor of the
    E packed experts; slots: device tensor of n_slots experts (or None for a
    planning-only cache); tables: device int32 tensor [n_layers][E] (or None)."""

    def __init__(self, shape: MoEShape, experts_host, slots, n_slots: int, tables):
        self._keep = list(experts_host)
        arr = (ctypes.c_void_p * len(self._keep))(*[_host_ptr(h) for h in self._keep])
        out = ctypes.c_void_p()
        _call(lib().ds_moe_cache_create, ctypes.byref(shape.c()), len(self._keep), arr, _ptr(slots), n_slots,
              _ptr(tables), ctypes.byref(out))
        self.handle = out

    def close(self):
        if self.handle:
            lib().ds_moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def layer(self, layer: int, weights: MoEWeights, x, out, workspace, stream=None, T: int | None = None):
        T = x.shape[0] if T is None else T
        _call(lib().ds_moe_cache_layer, self.handle, layer, ctypes.byref(weights.c()), x.data_ptr(), T,
              out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))

    def record(self, layer: int, counts):
        """Host policy step: counts a host int32 array [E]; returns the (slot,
        expert) fills it planned."""
        import numpy as np
        c = np.ascontiguousarray(counts, np.int32)
        fills = np.empty(2 * c.size, np.int32)
        n = ctypes.c_int32()
        rc = lib().ds_moe_cache_record(self.handle, layer, c.ctypes.data, fills.ctypes.data, ctypes.byref(n))
        if rc:
            raise DsMoeError(rc, "cache record")
        return [(int(fills[2 * j]), int(fills[2 * j + 1])) for j in range(n.value)]

    def slot(self, layer: int, expert: int) -> int:
        s = ctypes.c_int32()
        rc = lib().ds_moe_cache_slot(self.handle, layer, expert, ctypes.byref(s))
        if rc:
            raise DsMoeError(rc, "cache slot")
        return s.value

    def stats(self):
        h, m, r = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        lib().ds_moe_cache_stats(self.handle, ctypes.byref(h), ctypes.byref(m), ctypes.byref(r))
        return {"hits": h.value, "misses": m.value, "resident": r.value}


def _host_ptr(t):
    """Address of a host buffer: a torch tensor or a numpy array."""
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def stack(shape: MoEShape, layers, x, workspace, eps: float = 1e-6, stream=None, formats=None):
    """x[T][D] fp32 residual, updated in place through len(layers) layers.
    formats: optional per-layer expert formats (DS_Q2_K / DS_Q4_K)."""
    arr = (Weights * len(layers))(*[w.c() for w in layers])
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if formats is None:
        _call(lib().ds_moe_stack, ctypes.byref(shape.c()), arr, len(layers), x.data_ptr(),
              x.shape[0], eps, *ws, _stream(stream))
        return
    if len(formats) != len(layers):
        raise ValueError("one format per layer")
    fm = (ctypes.c_int32 * len(layers))(*formats)
    _call(lib().ds_moe_stack_mixed, ctypes.byref(shape.c()), arr, fm, len(layers), x.data_ptr(),
          x.shape[0], eps, *ws, _stream(stream))


def sync_status(stream=None):
    """Synchronise the stream and raise on a recorded device-side error."""
    _call(lib().ds_moe_sync_status, _stream(stream))
