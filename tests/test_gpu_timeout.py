"""A bounded device wait that runs out: the error path of the decode kernels.

Every wait in the persistent decode kernels is bounded.  When one expires the
kernel records ST_TIMEOUT in the device status word, waits (with the full
bound) for the bulk copies it has in flight, and returns, so the context
stays usable and the next call is unaffected.

A test build of the library (the same objects, except that the decode kernels
are compiled with DS_MOE_TEST_HOOKS) can hold the route back from the blocks
and shorten the bound to 1 ms, so that every wait for the route runs out; the
product library has no such hook.  Checks, on the one-token streaming kernel
and on the three-kernel chain: the held call reports DS_ERR_TIMEOUT through
ds_moe_sync_status well within the normal 2 s bound, and the next call with
the hook off gives the same output as before the held call, bit for bit (no
copy of the aborted call landed in a later one).  Nothing here faults the GPU:
the waits end by their bound and the kernels return normally.
"""
import ctypes
import time
from dataclasses import replace

import numpy as np
import pytest

import dsgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_quantized_routed_router_gb300 as ds  # noqa: E402
from bit_quantized_routed_router_gb300 import synthetic  # noqa: E402


@pytest.fixture(scope="module")
def hooks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_routed_router_gb300 import build
    L = ds.load(build.build_test_hooks())
    L.ds_moe_test_hooks.restype = ctypes.c_int
    L.ds_moe_test_hooks.argtypes = [ctypes.c_uint, ctypes.c_ulonglong]
    yield L
    L.ds_moe_test_hooks(0, 0)


def call(L, sh, W, x, out, ws):
    err = ctypes.create_string_buffer(512)
    rc = L.ds_moe_layer(ctypes.byref(sh.c()), ctypes.byref(W.c()), x.data_ptr(), x.shape[0], out.data_ptr(),
                        ws.data_ptr(), ws.numel(), None, None, err, 512)
    assert rc == ds.DS_OK, err.value
    t0 = time.perf_counter()
    rc = L.ds_moe_sync_status(None, err, 512)
    return rc, err.value.decode(), time.perf_counter() - t0


@pytest.mark.parametrize("T,path", [(1, ds.PATH_STREAM), (3, ds.PATH_DECODE3)])
def test_route_wait_runs_out_and_next_call_is_clean(hooks, T, path):
    cfg = replace(dsgen.TINY, name="timeout D=1024", T=T, D=1024, F=1024, E=16, k=4, Fs=512,
                  shared_sigma=0.02, x_dtype="bf16", router_dtype="bf16", router_sigma=0.02, seed=31)
    sh = synthetic.shape_of(cfg)
    assert ds.layer_path(sh, T) == path
    W = synthetic.build_layer(cfg)
    x = synthetic.build_x(cfg)
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, cfg.D), dtype=torch.float32, device="cuda")
    assert hooks.ds_moe_test_hooks(0, 0) == 0
    rc, msg, _ = call(hooks, sh, W, x, out, ws)
    assert rc == ds.DS_OK, msg
    ref = out.cpu().numpy().copy()
    assert np.isfinite(ref).all()

    assert hooks.ds_moe_test_hooks(1, 1_000_000) == 0  # hold the route; 1 ms bound
    out.fill_(float("nan"))
    rc, msg, dt = call(hooks, sh, W, x, out, ws)
    assert rc == ds.DS_ERR_TIMEOUT, (rc, msg)
    assert "timed out" in msg
    assert dt < 1.0, f"the held call took {dt:.2f} s: the shortened bound did not apply"

    assert hooks.ds_moe_test_hooks(0, 0) == 0
    for _ in range(2):
        rc, msg, _ = call(hooks, sh, W, x, out, ws)
        assert rc == ds.DS_OK, msg
        assert np.array_equal(out.cpu().numpy(), ref)
