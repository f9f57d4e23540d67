"""Seeded synthetic inputs for the routed-MoE layer (test and benchmark infrastructure).

Serves both the oracle and the CUDA path; holds none of the method's
arithmetic (no quantisation, routing or FFN).  The generator itself is
defined in ``gen/dsgen_core.h`` (Philox4x32-10, Irwin-Hall(8) normals);
host fills come from ``libdsgen_host.so`` and device fills from
``libdsgen_cuda.so`` and produce identical bits.

Workload shapes follow the pages: n_embd 4096, 256 routed experts, top-6,
one shared expert, expert FFN width 2048 ("Understanding Dwarf Star",
2.4.3 shape table; "The sparsity that pays for everything else in
DwarfStar", "Where the parameters actually are").
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
T_X, T_ROUTER_W, T_ZIPF_PERM = 1, 2, 3
T_SHARED_GATE, T_SHARED_UP, T_SHARED_DOWN = 4, 5, 6
T_EXPERT_GATE, T_EXPERT_UP, T_EXPERT_DOWN = 7, 8, 9

QK, QBYTES = 256, 84
BLOCK_BYTES = {"q2k": 84, "q4k": 144}  # bytes per 256-weight block of each expert format


@dataclass(frozen=True)
class Config:
    """One synthetic workload.  Sizes and value distributions as named."""
    name: str
    T: int
    D: int
    E: int
    k: int
    F: int
    Fs: int                 # shared expert width (0 = none)
    x_dtype: str            # "f32" | "bf16"
    router_dtype: str       # "f32" | "bf16"
    router_dist: str        # "normal" | "uniform" (both std router_sigma)
    router_sigma: float
    expert_sigma: float
    shared_sigma: float
    zipf_s: float           # 0 = no popularity bias
    seed: int
    layers: int = 1
    expert_fmt: str = "q2k"  # "q2k" | "q4k"

    def rows_blocks(self, in_dim: int) -> int:
        return (in_dim + QK - 1) // QK

    @property
    def block_bytes(self) -> int:
        return BLOCK_BYTES[self.expert_fmt]

    @property
    def expert_bytes(self) -> int:
        return self.block_bytes * (2 * self.F * self.rows_blocks(self.D) + self.D * self.rows_blocks(self.F))


TINY = Config("tiny T=8 D=256 E=16 k=2 F=128", 8, 256, 16, 2, 128, 0, "f32", "f32", "normal",
              0.05, 0.02, 0.0, 0.0, 0)
DECODE1 = Config("decode T=1 D=4096 E=256 k=6 F=2048 Fs=2048", 1, 4096, 256, 6, 2048, 2048,
                 "bf16", "bf16", "normal", 0.02, 0.02, 0.02, 0.0, 1)
DECODE32_ZIPF = Config("decode T=32 zipf(1.1) D=4096 E=256 k=6 F=2048 Fs=2048", 32, 4096, 256, 6,
                       2048, 2048, "bf16", "bf16", "normal", 0.02, 0.02, 0.02, 1.1, 2)
PREFILL = Config("prefill T=4096 D=4096 E=256 k=6 F=2048 Fs=2048", 4096, 4096, 256, 6, 2048,
                 2048, "bf16", "bf16", "uniform", 0.02, 0.02, 0.02, 0.0, 3)
PREFILL_ZIPF = replace(PREFILL, name="prefill T=4096 zipf(1.1) D=4096 E=256 k=6 F=2048 Fs=2048",
                       zipf_s=1.1)
STACK = Config("stack 43 layers T=8 D=4096 E=256 k=6 F=2048 Fs=2048", 8, 4096, 256, 6, 2048,
               2048, "bf16", "bf16", "normal", 0.02, 0.02, 0.02, 0.0, 4, layers=43)

DECODE1_Q4K = replace(DECODE1, name="decode T=1 Q4_K experts D=4096 E=256 k=6 F=2048 Fs=2048",
                      expert_fmt="q4k")

ALL = [TINY, DECODE1, DECODE32_ZIPF, PREFILL, PREFILL_ZIPF, STACK]


# ------------------------------------------------------------------ build --

def build(force: bool = False) -> None:
    """Compile the host fill library (gcc) and, if nvcc exists, the device fills."""
    host = os.path.join(HERE, "libdsgen_host.so")
    src = os.path.join(HERE, "dsgen_host.c")
    hdr = os.path.join(HERE, "dsgen_core.h")
    if force or _stale(host, [src, hdr]):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", host,
                               src, "-lpthread", "-lm"])
    dev = os.path.join(HERE, "libdsgen_cuda.so")
    dsrc = os.path.join(HERE, "dsgen_cuda.cu")
    if force or _stale(dev, [dsrc, hdr]):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-o", dev, dsrc])


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        path = os.path.join(HERE, "libdsgen_host.so")
        if not os.path.exists(path):
            build()
        L = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32 = ctypes.c_uint32
        L.dsgen_scale_normal.restype = ctypes.c_float
        L.dsgen_scale_normal.argtypes = [ctypes.c_double]
        L.dsgen_scale_uniform.restype = ctypes.c_float
        L.dsgen_scale_uniform.argtypes = [ctypes.c_double]
        for fn in (L.dsgen_fill_normal, L.dsgen_fill_uniform):
            fn.restype = None
            fn.argtypes = [f32p, u16p, ctypes.c_uint64, u32, u32, u32, u32, ctypes.c_uint64,
                           ctypes.c_float, ctypes.c_int]
        L.dsgen_x_rows.restype = None
        L.dsgen_x_rows.argtypes = [f32p, u16p, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.POINTER(ctypes.c_int32), u32, u32, ctypes.c_float]
        L.dsgen_zipf_ranks.restype = None
        L.dsgen_zipf_ranks.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, u32, u32]
        L.dsgen_philox.restype = None
        L.dsgen_philox.argtypes = [u32] * 6 + [ctypes.POINTER(ctypes.c_uint32)]
        _host = L
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        path = os.path.join(HERE, "libdsgen_cuda.so")
        if not os.path.exists(path):
            build()
        L = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        u32 = ctypes.c_uint32
        L.dsgen_cuda_fill.restype = ctypes.c_int
        L.dsgen_cuda_fill.argtypes = [vp, vp, ctypes.c_uint64, u32, u32, u32, u32, ctypes.c_uint64,
                                      ctypes.c_float, ctypes.c_int, vp]
        L.dsgen_cuda_x_rows.restype = ctypes.c_int
        L.dsgen_cuda_x_rows.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int64, vp, u32, u32,
                                        ctypes.c_float, vp]
        _dev = L
    return _dev


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct)) if a is not None else None


def scale_normal(sigma: float) -> float:
    return host_lib().dsgen_scale_normal(sigma)


def scale_uniform(a: float) -> float:
    return host_lib().dsgen_scale_uniform(a)


def philox(c, k):
    out = (ctypes.c_uint32 * 4)()
    host_lib().dsgen_philox(c[0], c[1], c[2], c[3], k[0], k[1], out)
    return list(out)


# ------------------------------------------------------------ host fills --

def host_fill(n, seed, layer, tensor, sub, sigma, dist="normal", idx0=0, bf16=False, nthreads=None):
    """n generated fp32 values (and their bf16 bit patterns if bf16=True)."""
    nthreads = nthreads or os.cpu_count() or 1
    out = np.empty(n, np.float32)
    ob = np.empty(n, np.uint16) if bf16 else None
    L = host_lib()
    if dist == "normal":
        L.dsgen_fill_normal(_p(out, ctypes.c_float), _p(ob, ctypes.c_uint16), n, seed, layer, tensor,
                            sub, idx0, scale_normal(sigma), nthreads)
    else:  # uniform with standard deviation sigma: half-width sigma*sqrt(3)
        L.dsgen_fill_uniform(_p(out, ctypes.c_float), _p(ob, ctypes.c_uint16), n, seed, layer, tensor,
                             sub, idx0, scale_uniform(sigma * math.sqrt(3.0)), nthreads)
    return (out, ob) if bf16 else out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def host_x(cfg: Config, attempts=None, layer=0, T=None):
    """Activations [T][D]: fp32 values for "f32" configs, bf16 bits for "bf16"."""
    T = cfg.T if T is None else T
    att = None if attempts is None else np.ascontiguousarray(attempts, np.int32)
    out = np.empty((T, cfg.D), np.float32)
    ob = np.empty((T, cfg.D), np.uint16) if cfg.x_dtype == "bf16" else None
    host_lib().dsgen_x_rows(_p(out, ctypes.c_float), _p(ob, ctypes.c_uint16), T, cfg.D,
                            _p(att, ctypes.c_int32), cfg.seed, layer, scale_normal(1.0))
    return ob if ob is not None else out


def host_router(cfg: Config, layer=0):
    """Router weights [E][D]: fp32 values or bf16 bits per router_dtype."""
    n = cfg.E * cfg.D
    r = host_fill(n, cfg.seed, layer, T_ROUTER_W, 0, cfg.router_sigma, cfg.router_dist,
                  bf16=cfg.router_dtype == "bf16")
    if cfg.router_dtype == "bf16":
        return r[1].reshape(cfg.E, cfg.D)
    return r.reshape(cfg.E, cfg.D)


def host_bias(cfg: Config, layer=0):
    """Per-expert popularity bias (fp32 [E]) or None: bias_e = -s*ln(rank_e),
    ranks a seeded shuffle of 1..E, so softmax mass ~ rank^-s (Zipf(s))."""
    if cfg.zipf_s == 0.0:
        return None
    rank = np.empty(cfg.E, np.int32)
    host_lib().dsgen_zipf_ranks(_p(rank, ctypes.c_int32), cfg.E, cfg.seed, layer)
    return np.array([-cfg.zipf_s * math.log(float(r)) for r in rank], np.float32)


def host_shared(cfg: Config, layer=0):
    """Shared expert bf16 bits: gate [Fs][D], up [Fs][D], down [D][Fs]."""
    if cfg.Fs == 0:
        return None
    out = []
    for t, shape in ((T_SHARED_GATE, (cfg.Fs, cfg.D)), (T_SHARED_UP, (cfg.Fs, cfg.D)),
                     (T_SHARED_DOWN, (cfg.D, cfg.Fs))):
        _, b = host_fill(shape[0] * shape[1], cfg.seed, layer, t, 0, cfg.shared_sigma, bf16=True)
        out.append(b.reshape(shape))
    return out


def host_expert_f32(cfg: Config, e: int, layer=0):
    """Routed expert e's fp32 weights: gate [F][D], up [F][D], down [D][F]."""
    g = host_fill(cfg.F * cfg.D, cfg.seed, layer, T_EXPERT_GATE, e, cfg.expert_sigma).reshape(cfg.F, cfg.D)
    u = host_fill(cfg.F * cfg.D, cfg.seed, layer, T_EXPERT_UP, e, cfg.expert_sigma).reshape(cfg.F, cfg.D)
    d = host_fill(cfg.D * cfg.F, cfg.seed, layer, T_EXPERT_DOWN, e, cfg.expert_sigma).reshape(cfg.D, cfg.F)
    return g, u, d


# ----------------------------------------------------------- device fills --

def _check(rc):
    if rc != 0:
        raise RuntimeError(f"dsgen cuda error {rc}")


def dev_fill(out_f32, out_bf16, n, seed, layer, tensor, sub, sigma, dist="normal", stream=0):
    """Fill device buffers (torch tensors or None) with the same values as host_fill."""
    f = out_f32.data_ptr() if out_f32 is not None else None
    b = out_bf16.data_ptr() if out_bf16 is not None else None
    if dist == "normal":
        c, uni = scale_normal(sigma), 0
    else:
        c, uni = scale_uniform(sigma * math.sqrt(3.0)), 1
    _check(dev_lib().dsgen_cuda_fill(f, b, n, seed, layer, tensor, sub, 0, c, uni, stream))


def dev_x(cfg: Config, out_f32, out_bf16, attempts=None, layer=0, T=None, stream=0):
    T = cfg.T if T is None else T
    a = attempts.data_ptr() if attempts is not None else None
    _check(dev_lib().dsgen_cuda_x_rows(out_f32.data_ptr() if out_f32 is not None else None,
                                       out_bf16.data_ptr() if out_bf16 is not None else None,
                                       T, cfg.D, a, cfg.seed, layer, scale_normal(1.0), stream))
