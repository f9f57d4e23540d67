"""A token whose activations are NaN, on every kernel path.

Its router logits are all NaN, so no expert is a candidate for any of its k
picks: the selection takes expert 0 for each (an id that is always in range),
flags the status word, and ds_moe_sync_status reports DS_ERR_DEVICE_CHECK.
The next call on clean input must then be bit-identical to the same clean call
made before, which shows that nothing the bad call left in the workspace or
the status word leaks into it.
"""
from dataclasses import replace

import pytest

import dsgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_quantized_routed_router_gb300 as ds  # noqa: E402
from bit_quantized_routed_router_gb300 import synthetic  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_routed_router_gb300 import build
    build.build()
    yield


def _w1024(T, Fs):
    return replace(dsgen.TINY, name=f"D=1024 E=16 k=4 T={T} Fs={Fs}", T=T, D=1024, F=1024, E=16, k=4,
                   Fs=Fs, shared_sigma=0.02, x_dtype="bf16", router_dtype="bf16", router_sigma=0.02, seed=5)


CASES = [(_w1024(1, 512), ds.PATH_STREAM), (_w1024(3, 512), ds.PATH_DECODE3),
         (_w1024(8, 1024), ds.PATH_BATCHED_DECODE), (_w1024(64, 1024), ds.PATH_TENSOR_CORE),
         (_w1024(300, 1024), ds.PATH_TENSOR_CORE), (dsgen.TINY, ds.PATH_GROUPED_GEMV)]


@pytest.mark.parametrize("cfg,path", CASES, ids=["stream", "chain", "batched", "tc64", "tc300", "gemv"])
def test_nan_token_is_reported_and_the_next_call_is_clean(cfg, path):
    sh = synthetic.shape_of(cfg)
    W = synthetic.build_layer(cfg)
    x = synthetic.build_x(cfg)
    assert ds.layer_path(sh, cfg.T, x) == path
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device="cuda")
    out = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device="cuda")
    ds.layer(sh, W, x, out, ws)
    ds.sync_status()
    ref = out.cpu().clone()
    assert torch.isfinite(ref).all()

    bad = x.clone()
    # bf16 activations are held as their 16-bit patterns: 0x7FC0 is a quiet NaN
    bad[cfg.T // 2] = float("nan") if bad.is_floating_point() else 0x7FC0
    ds.layer(sh, W, bad, out, ws)
    with pytest.raises(ds.DsMoeError) as ei:
        ds.sync_status()
    assert ei.value.code == ds.DS_ERR_DEVICE_CHECK
    ds.sync_status()  # read and cleared

    out.fill_(7.0)
    ds.layer(sh, W, x, out, ws)
    ds.sync_status()
    assert torch.equal(out.cpu(), ref)
