"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/ds_moe.h declares, sizes its buffers as the block
format fixes, and rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import bit_quantized_routed_router_gb300 as ds
from bit_quantized_routed_router_gb300 import build as dsbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    dsbuild.build()
    return ds.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "ds_moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_moe_\w+)\s*\(", txt)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(ds.SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", ds.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (ds_moe_\w+)$", out, flags=re.M))
    for s in declared_symbols():
        assert s in exported, s
        assert hasattr(L, s)


def test_sizes(L):
    assert ds.q2k_bytes(1, 256) == 84
    assert ds.q2k_bytes(2048, 4096) == 2048 * 16 * 84
    assert ds.q2k_bytes(4096, 128) == 4096 * 84  # zero-padded rows
    assert ds.q2k_bytes(-1, 256) == 0
    assert ds.expert_bytes(4096, 2048) == 8_257_536
    assert ds.expert_bytes(256, 128) == 84 * (2 * 128 + 256)
    assert ds.version().startswith("ds_moe")
    assert ds.q4k_bytes(1, 256) == 144
    assert ds.q4k_bytes(4096, 128) == 4096 * 144
    assert ds.q4k_bytes(3, -1) == 0
    assert ds.expert_bytes(4096, 2048, ds.DS_Q4_K) == 3 * 2048 * 16 * 144
    assert ds.expert_bytes(256, 128, ds.DS_Q4_K) == 144 * (2 * 128 + 256)
    assert ds.expert_bytes(4096, 2048, 7) == 0


def test_workspace_bytes_and_validation(L):
    sh = ds.MoEShape(4096, 256, 2048, 2048, 6)
    ws1 = ds.workspace_bytes(sh, 1)
    ws32 = ds.workspace_bytes(sh, 32)
    assert 0 < ws1 < ws32
    assert ds.workspace_bytes(sh, 0) > 0
    bad = [ds.MoEShape(4000, 256, 2048, 2048, 6), ds.MoEShape(4096, 0, 2048, 2048, 6),
           ds.MoEShape(4096, 256, 2000, 2048, 6), ds.MoEShape(4096, 256, 2048, 100, 6),
           ds.MoEShape(4096, 256, 2048, 2048, 0), ds.MoEShape(4096, 4, 2048, 2048, 5),
           ds.MoEShape(4096, 256, 2048, 2048, 6, x_dtype=7),
           ds.MoEShape(4096, 256, 2048, 2048, 6, routed_scale=float("nan")),
           ds.MoEShape(4096, 256, 2048, 2048, 6, logit_scale=-1.0),
           ds.MoEShape(4096, 256, 2048, 2048, 6, logit_scale=float("inf")),
           ds.MoEShape(4096, 256, 2048, 2048, 6, bias_select_only=2),
           ds.MoEShape(4096, 256, 2048, 2048, 6, expert_format=2),
           ds.MoEShape(4096, 256, 2048, 2048, 6, expert_format=-1)]
    for b in bad:
        with pytest.raises(ds.DsMoeError) as ei:
            ds.workspace_bytes(b, 4)
        assert ei.value.code in (ds.DS_ERR_INVALID_ARG, ds.DS_ERR_UNSUPPORTED)
    with pytest.raises(ds.DsMoeError):
        ds.workspace_bytes(sh, -1)


def test_layer_rejects_bad_arguments_on_host(L):
    sh = ds.MoEShape(256, 16, 128, 0, 2, ds.DS_F32, ds.DS_F32).c()
    err = ctypes.create_string_buffer(256)
    # missing weights struct
    rc = L.ds_moe_layer(ctypes.byref(sh), None, 16, 8, 16, 256, 1 << 20, None, None, err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG and b"weights" in err.value
    # misaligned expert blob
    w = ds.Weights(256, None, None, None, None, 0x1001)
    rc = L.ds_moe_layer(ctypes.byref(sh), ctypes.byref(w), 256, 8, 256, 256, 1 << 20, None, None,
                        err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG and b"aligned" in err.value
    # workspace too small
    w = ds.Weights(256, None, None, None, None, 0x1000)
    rc = L.ds_moe_layer(ctypes.byref(sh), ctypes.byref(w), 256, 8, 256, 256, 16, None, None, err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG and b"workspace too small" in err.value
    # T == 0 is a no-op and touches nothing
    rc = L.ds_moe_layer(ctypes.byref(sh), ctypes.byref(w), None, 0, None, None, 0, None, None, err, 256)
    assert rc == ds.DS_OK
    # shared expert declared but missing
    sh2 = ds.MoEShape(256, 16, 128, 128, 2, ds.DS_F32, ds.DS_F32).c()
    rc = L.ds_moe_layer(ctypes.byref(sh2), ctypes.byref(w), 256, 8, 256, 256, 1 << 30, None, None,
                        err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG and b"shared" in err.value
    # the stack wants bf16 normalised inputs
    rc = L.ds_moe_stack(ctypes.byref(sh), ctypes.byref(w), 1, 256, 8, 1e-6, 256, 1 << 30, None,
                        err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG


def test_quantize_rejects_bad_arguments_on_host(L):
    err = ctypes.create_string_buffer(256)
    assert L.ds_moe_quantize_q2k(None, 4, 256, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
    assert L.ds_moe_quantize_q2k(16, -1, 256, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
    assert L.ds_moe_quantize_q2k(18, 4, 256, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
    assert L.ds_moe_quantize_q2k(16, 0, 256, 16, None, err, 256) == ds.DS_OK
    for q in (L.ds_moe_quantize_q4k, L.ds_moe_quantize_q2k):
        assert q(None, 4, 256, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
        assert q(16, 4, -2, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
        assert q(16, 4, 256, 17, None, err, 256) == ds.DS_ERR_INVALID_ARG   # out not 4-byte aligned
        assert q(16, 4, 0, 16, None, err, 256) == ds.DS_OK                  # nothing to do
    for dq in (L.ds_moe_dequantize_q4k, L.ds_moe_dequantize_q2k):
        assert dq(16, 4, 256, None, None, err, 256) == ds.DS_ERR_INVALID_ARG
        assert dq(16, 4, 256, 18, None, err, 256) == ds.DS_ERR_INVALID_ARG
        assert dq(16, -4, 256, 16, None, err, 256) == ds.DS_ERR_INVALID_ARG
        assert dq(16, 0, 256, 16, None, err, 256) == ds.DS_OK


def test_layer_path_host_checks(L):
    sh = ds.MoEShape(4096, 256, 2048, 2048, 6)
    assert ds.layer_path(sh, 0) == ds.PATH_NONE
    # 8 tokens: the batched decode kernels where the device has them (and the
    # CUDA driver can build tensor maps), the grouped GEMV path on a host
    # without a GPU
    import torch
    gpu = torch.cuda.is_available()
    assert ds.layer_path(sh, 8) == (ds.PATH_BATCHED_DECODE if gpu else ds.PATH_GROUPED_GEMV)
    assert ds.layer_path(sh, 3) == ds.PATH_DECODE3
    with pytest.raises(ds.DsMoeError):
        ds.layer_path(ds.MoEShape(4000, 256, 2048, 2048, 6), 4)
    with pytest.raises(ds.DsMoeError):
        ds.layer_path(sh, -1)
    # Q4_K experts: the streaming kernel for one token where a device can run
    # it (else the three-kernel chain), the chain up to four tokens, the
    # tensor cores beyond (the grouped GEMV path without a device)
    q4 = ds.MoEShape(4096, 256, 2048, 2048, 6, expert_format=ds.DS_Q4_K)
    assert ds.layer_path(q4, 1) == (ds.PATH_STREAM if gpu else ds.PATH_DECODE3)
    for T in (2, 4):
        assert ds.layer_path(q4, T) == ds.PATH_DECODE3
    for T in (8, 4096):
        assert ds.layer_path(q4, T) == (ds.PATH_TENSOR_CORE if gpu else ds.PATH_GROUPED_GEMV)


def test_stack_mixed_rejects_bad_format_before_launch(L):
    """The per-layer format list is checked on the host: nothing runs."""
    sh = ds.MoEShape(4096, 256, 2048, 2048, 6).c()
    W = (ds.Weights * 2)()
    err = ctypes.create_string_buffer(256)
    fm = (ctypes.c_int32 * 2)(0, 5)
    rc = L.ds_moe_stack_mixed(ctypes.byref(sh), W, fm, 2, 256, 8, 1e-6, 256, 1 << 30, None, err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG and b"formats[1]" in err.value
    shf = ds.MoEShape(4096, 256, 2048, 2048, 6, x_dtype=ds.DS_F32).c()
    fm_ok = (ctypes.c_int32 * 2)(0, 1)
    rc = L.ds_moe_stack_mixed(ctypes.byref(shf), W, fm_ok, 2, 256, 8, 1e-6, 256, 1 << 30, None, err, 256)
    assert rc == ds.DS_ERR_INVALID_ARG
