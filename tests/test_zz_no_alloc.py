"""ds_moe_layer_noalloc: the layer for callers that cannot allocate device
memory where they run it (a plugin whose host program owns all device
memory, a real-time loop that must not take cudaMalloc's device-wide
synchronisation).  Its scratch is a static device array inside the library,
so the caller passes only inputs and outputs.

The check: it runs the same kernels as ds_moe_layer (caller workspace) on the
same inputs, so its output must equal that one bit for bit, on two calls in a
row (the second with another batch and another path, so contents left in the
shared array by the first call must not matter); a batch too large for the
static array is refused with a clear error, and T == 0 with missing weights is
rejected as ds_moe_layer rejects it.

This file is collected last on purpose; it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest

import dsgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_quantized_routed_router_gb300 as ds  # noqa: E402
from bit_quantized_routed_router_gb300 import synthetic  # noqa: E402

@pytest.fixture(scope="module")
def layer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_routed_router_gb300 import build
    build.build()
    cfg = dsgen.DECODE1
    return cfg, synthetic.build_layer(cfg)


def with_workspace(cfg, W, x):
    sh = synthetic.shape_of(cfg)
    ws = torch.empty(ds.workspace_bytes(sh, x.shape[0]), dtype=torch.uint8, device="cuda")
    out = torch.empty((x.shape[0], cfg.D), dtype=torch.float32, device="cuda")
    ds.layer(sh, W, x, out, ws)
    ds.sync_status()
    return out.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice(layer):
    cfg, W = layer
    sh = synthetic.shape_of(cfg)
    from dataclasses import replace
    for T, seed_layer in ((8, 0), (1, 3)):  # two calls in a row, different batches and paths
        c = replace(cfg, T=T)
        x = synthetic.build_x(c, layer=seed_layer)
        ref = with_workspace(c, W, x)
        out = torch.full((T, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
        ds.layer_noalloc(sh, W, x, out)
        ds.sync_status()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert np.array_equal(got, ref), f"T={T}: differs from ds_moe_layer"
        rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
        assert rms > 0


def test_noalloc_zero_tokens_validates_weights(layer):
    cfg, W = layer
    sh = synthetic.shape_of(cfg)
    bad = ds.MoEWeights(router_w=None, experts=None)
    x = torch.zeros((1, cfg.D), dtype=torch.int16, device="cuda")
    out = torch.zeros((1, cfg.D), dtype=torch.float32, device="cuda")
    for fn in (lambda: ds.layer_noalloc(sh, bad, x, out, T=0),
               lambda: ds.layer(sh, bad, x, out, torch.empty(256, dtype=torch.uint8, device="cuda"), T=0)):
        with pytest.raises(ds.DsMoeError) as ei:
            fn()
        assert ei.value.code == ds.DS_ERR_INVALID_ARG
    ds.layer_noalloc(sh, W, x, out, T=0)  # a valid call with no tokens does nothing
    ds.sync_status()


def test_noalloc_refuses_batches_beyond_its_scratch(layer):
    cfg, W = layer
    sh = synthetic.shape_of(cfg)
    T = 1024  # needs far more scratch at this shape than the static 64 MiB
    assert ds.workspace_bytes(sh, T) > 64 << 20
    fits = [t for t in (8, 32, 128, 192, 256) if ds.workspace_bytes(sh, t) <= 64 << 20]
    print(f"batches that fit the static scratch: {fits}")
    x = torch.zeros((T, cfg.D), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, cfg.D), dtype=torch.float32, device="cuda")
    with pytest.raises(ds.DsMoeError) as ei:
        ds.layer_noalloc(sh, W, x, out)
    assert ei.value.code == ds.DS_ERR_INVALID_ARG
    assert "static scratch" in str(ei.value)
    ds.sync_status()
