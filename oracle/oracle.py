"""Python front of the fp64 CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product package.
It shares no code with the CUDA path; both sides read the same seeded inputs
from ``gen/dsgen.py``, which holds none of the method's arithmetic.

What each function computes is stated, with the pages it follows, in the C
source.  This module only marshals arrays and drives the regeneration of the
experts a routing decision actually selects, so full-size layers never have
to be materialised on the host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(os.path.dirname(HERE), "gen"))
import dsgen  # noqa: E402

LIB = os.path.join(HERE, "liboracle.so")
SRC = os.path.join(HERE, "oracle.c")
NTHREADS = os.cpu_count() or 1


def build(force: bool = False) -> None:
    """Compile the oracle with gcc.  -ffp-contract=off keeps every a*b+c as a
    rounded multiply then a rounded add on every host (aarch64 gcc would
    otherwise fuse them)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", LIB, SRC, "-lpthread", "-lm"])


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
        L.oracle_fp16_value.restype = dbl
        L.oracle_fp16_value.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_round.restype = ctypes.c_uint16
        L.oracle_bf16_round.argtypes = [dbl]
        L.oracle_q2k_bytes.restype = i64
        L.oracle_q2k_bytes.argtypes = [i64, i64]
        L.oracle_expert_bytes.restype = i64
        L.oracle_expert_bytes.argtypes = [i64, i64]
        L.oracle_q2k_quantize.restype = ctypes.c_int
        L.oracle_q2k_quantize.argtypes = [vp, i64, i64, vp, ctypes.c_int]
        L.oracle_q2k_dequantize.restype = None
        L.oracle_q2k_dequantize.argtypes = [vp, i64, i64, vp]
        L.oracle_q4k_bytes.restype = i64
        L.oracle_q4k_bytes.argtypes = [i64, i64]
        L.oracle_q4k_quantize.restype = ctypes.c_int
        L.oracle_q4k_quantize.argtypes = [vp, i64, i64, vp, ctypes.c_int]
        L.oracle_q4k_dequantize.restype = None
        L.oracle_q4k_dequantize.argtypes = [vp, i64, i64, vp]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [vp, i64, i64, vp, i64, vp, vp]
        L.oracle_select.restype = None
        L.oracle_select.argtypes = [vp, i64, i64, i32, dbl, dbl, vp, vp, vp]
        L.oracle_route.restype = None
        L.oracle_route.argtypes = [vp, i64, i32, i64, vp, vp, vp, vp]
        L.oracle_expert_bytes_fmt.restype = i64
        L.oracle_expert_bytes_fmt.argtypes = [ctypes.c_int, i64, i64]
        L.oracle_moe_layer_fmt.restype = ctypes.c_int
        L.oracle_moe_layer_fmt.argtypes = [ctypes.c_int, i64, i64, i64, i64, i64, i32, vp, vp, vp,
                                           vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
        L.oracle_moe_layer.restype = ctypes.c_int
        L.oracle_moe_layer.argtypes = [i64, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, ctypes.c_int]
        L.oracle_rmsnorm_bf16.restype = None
        L.oracle_rmsnorm_bf16.argtypes = [vp, i64, i64, dbl, vp]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# -------------------------------------------------------------- primitives --

def fp16_value(bits: int) -> float:
    return lib().oracle_fp16_value(bits)


def bf16_round(v: float) -> int:
    return lib().oracle_bf16_round(v)


def q2k_bytes(rows: int, in_dim: int) -> int:
    return lib().oracle_q2k_bytes(rows, in_dim)


def quantize(w: np.ndarray) -> np.ndarray:
    """Q2_K blocks of a [rows][in_dim] fp32 matrix, uint8 [rows][nb*84]."""
    w = _c(w, np.float32)
    rows, in_dim = w.shape
    out = np.zeros(q2k_bytes(rows, in_dim), np.uint8)
    if lib().oracle_q2k_quantize(_ptr(w), rows, in_dim, _ptr(out), NTHREADS):
        raise ValueError("Q2_K quantiser: non-finite or out-of-range input")
    return out.reshape(rows, -1)


def dequantize(q: np.ndarray, rows: int, in_dim: int) -> np.ndarray:
    q = _c(q, np.uint8)
    out = np.empty((rows, in_dim), np.float64)
    lib().oracle_q2k_dequantize(_ptr(q), rows, in_dim, _ptr(out))
    return out


def q4k_bytes(rows: int, in_dim: int) -> int:
    return lib().oracle_q4k_bytes(rows, in_dim)


def quantize_q4k(w: np.ndarray) -> np.ndarray:
    """Q4_K blocks of a [rows][in_dim] fp32 matrix, uint8 [rows][nb*144]."""
    w = _c(w, np.float32)
    rows, in_dim = w.shape
    out = np.zeros(q4k_bytes(rows, in_dim), np.uint8)
    if lib().oracle_q4k_quantize(_ptr(w), rows, in_dim, _ptr(out), NTHREADS):
        raise ValueError("Q4_K quantiser: non-finite or out-of-range input")
    return out.reshape(rows, -1)


def dequantize_q4k(q: np.ndarray, rows: int, in_dim: int) -> np.ndarray:
    q = _c(q, np.uint8)
    out = np.empty((rows, in_dim), np.float64)
    lib().oracle_q4k_dequantize(_ptr(q), rows, in_dim, _ptr(out))
    return out


def router_logits(x: np.ndarray, wr: np.ndarray, bias=None) -> np.ndarray:
    x, wr = _c(x, np.float64), _c(wr, np.float64)
    T, D = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float64)
    out = np.empty((T, E), np.float64)
    lib().oracle_router_logits(_ptr(x), T, D, _ptr(wr), E, _ptr(b), _ptr(out))
    return out


def select(logits: np.ndarray, k: int, routed_scale: float = 1.0, logit_scale: float = 1.0,
           unbias=None):
    """unbias: the router bias the logits include, when it is to steer the
    selection only (the weights then use the logits without it)."""
    L = _c(logits, np.float64)
    T, E = L.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    ub = None if unbias is None else _c(unbias, np.float64)
    lib().oracle_select(_ptr(L), T, E, k, routed_scale, logit_scale, None if ub is None else _ptr(ub),
                        _ptr(ids), _ptr(w))
    return ids, w


def route(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pos = np.empty(T * k, np.int32)
    lib().oracle_route(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(pos))
    return counts, offsets, perm, pos


FORMATS = {"q2k": 0, "q4k": 1}


def moe_layer(x, experts, shared, ids, w, D, E, F, Fs, want_parts=False, fmt="q2k"):
    """out[T][D] fp64.  experts: dict e -> packed uint8 blob (gate|up|down) in
    format fmt ("q2k" | "q4k"); shared: (gate, up, down) fp64 arrays or None."""
    x = _c(x, np.float64)
    T = x.shape[0]
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    w = _c(w, np.float64)
    keep = [None] * E
    ptrs = (ctypes.c_void_p * E)()
    for e, blob in experts.items():
        keep[e] = _c(blob, np.uint8)
        ptrs[e] = keep[e].ctypes.data
    if shared is not None:
        sg, su, sd = (_c(a, np.float64) for a in shared)
    else:
        sg = su = sd = None
    out = np.empty((T, D), np.float64)
    yp = np.empty((T * k, D), np.float64) if want_parts else None
    ys = np.empty((T, D), np.float64) if want_parts else None
    rc = lib().oracle_moe_layer_fmt(FORMATS[fmt], T, D, E, F, Fs, k, _ptr(x),
                                    ctypes.cast(ptrs, ctypes.c_void_p), _ptr(sg), _ptr(su),
                                    _ptr(sd), _ptr(ids), _ptr(w), _ptr(out), _ptr(yp), _ptr(ys),
                                    NTHREADS)
    if rc:
        raise ValueError("oracle_moe_layer: a selected expert has no weights")
    return (out, yp, ys) if want_parts else out


def rmsnorm_bf16(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = _c(x, np.float32)
    T, D = x.shape
    out = np.empty((T, D), np.uint16)
    lib().oracle_rmsnorm_bf16(_ptr(x), T, D, eps, _ptr(out))
    return out


# ------------------------------------------------------ workload drivers --

def as_f64(a, dtype: str) -> np.ndarray:
    """Exact fp64 values of generated inputs (bf16 bits or fp32)."""
    if dtype == "bf16":
        return dsgen.bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, np.float32).astype(np.float64)


def expert_blob(cfg: dsgen.Config, e: int, layer: int = 0) -> np.ndarray:
    """Expert e regenerated from its counters and packed by the oracle's quantiser
    in the workload's expert format."""
    g, u, d = dsgen.host_expert_f32(cfg, e, layer)
    q = quantize_q4k if cfg.expert_fmt == "q4k" else quantize
    return np.concatenate([q(g).ravel(), q(u).ravel(), q(d).ravel()])


class LayerOracle:
    """Oracle for one synthetic layer of a workload (weights regenerated on demand)."""

    def __init__(self, cfg: dsgen.Config, layer: int = 0):
        self.cfg, self.layer = cfg, layer
        self.wr = as_f64(dsgen.host_router(cfg, layer), cfg.router_dtype)
        b = dsgen.host_bias(cfg, layer)
        self.bias = None if b is None else b.astype(np.float64)
        sh = dsgen.host_shared(cfg, layer)
        self.shared = None if sh is None else [as_f64(a, "bf16") for a in sh]
        self._experts = {}

    def logits(self, x64):
        return router_logits(x64, self.wr, self.bias)

    def experts(self, ids):
        need = sorted(set(int(e) for e in np.asarray(ids).ravel()))
        for e in need:
            if e not in self._experts:
                self._experts[e] = expert_blob(self.cfg, e, self.layer)
        return {e: self._experts[e] for e in need}

    def forward(self, x64, want_parts=False):
        """(out, ids, w, logits) for activations x64 [n][D] (exact fp64 values)."""
        c = self.cfg
        L = self.logits(x64)
        ids, w = select(L, c.k)
        res = moe_layer(x64, self.experts(ids), self.shared, ids, w, c.D, c.E, c.F, c.Fs,
                        want_parts=want_parts, fmt=c.expert_fmt)
        return res, ids, w, L


def min_top_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: smallest gap between consecutive logits among the top k+1."""
    s = -np.sort(-logits, axis=1)[:, : min(k + 1, logits.shape[1])]
    if s.shape[1] < 2:
        return np.full(logits.shape[0], np.inf)
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


GAP = 1e-4


def resample_attempts(cfg: dsgen.Config, lo: LayerOracle, tokens=None, max_attempts=64):
    """Resample-attempt counter per token so that no two of the top k+1 logits
    lie within GAP of each other (oracle fp64), which makes the selected ids
    and their order one unique answer at fp32 too.  Returns int32 [T]."""
    T = cfg.T
    att = np.zeros(T, np.int32)
    todo = np.arange(T) if tokens is None else np.asarray(tokens)
    for _ in range(max_attempts):
        x = as_f64(dsgen.host_x(cfg, att, lo.layer), cfg.x_dtype)
        gaps = min_top_gap(lo.logits(x[todo]), cfg.k)
        bad = todo[gaps < GAP]
        if bad.size == 0:
            return att
        att[bad] += 1
        todo = bad
    raise RuntimeError("resampling did not converge")
