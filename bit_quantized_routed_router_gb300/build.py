"""Build the ds_moe CUDA library in-tree for sm_103a (nvcc, no cmake).

Each translation unit is compiled in parallel, then linked into
``bit_quantized_routed_router_gb300/libds_moe.so``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libds_moe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "-I", os.path.join(ROOT, "include")]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(ROOT, "include", "ds_moe.h")]


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def _compile(src, extra, suffix=""):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + suffix + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest([src] + headers()):
        return obj
    cmd = ["nvcc"] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < _newest(objs):
        cmd = ["nvcc"] + ARCH + ["-shared", "-o", LIB] + objs
        subprocess.check_call(cmd)
    return LIB


HOOKS_LIB = os.path.join(BUILD, "libds_moe_test_hooks.so")


def build_test_hooks() -> str:
    """A second library for the tests only: the same objects, except that the
    decode kernels are compiled with DS_MOE_TEST_HOOKS (a hook that holds the
    route so that the device waits for it run out, and ds_moe_test_hooks to
    set it).  The product library never contains the hook."""
    build()
    srcs = sources()
    objs = []
    for s in srcs:
        if os.path.basename(s) == "decode_fast.cu":
            objs.append(_compile(s, ["-DDS_MOE_TEST_HOOKS"], suffix="_hooks"))
        else:
            objs.append(os.path.join(BUILD, os.path.basename(s)[:-3] + ".o"))
    if not os.path.exists(HOOKS_LIB) or os.path.getmtime(HOOKS_LIB) < _newest(objs):
        subprocess.check_call(["nvcc"] + ARCH + ["-shared", "-o", HOOKS_LIB] + objs)
    return HOOKS_LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
