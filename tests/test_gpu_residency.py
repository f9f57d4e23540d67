"""Expert residency beyond device memory, on the GPU.

"Page the experts off the SSD" ("The cache is never allowed to become a
correctness structure"): whatever the cache holds, the layer's output is the
same.  Here the routed experts live in pinned host memory and a slot table
says which of them also sit in device slots; the kernels read an expert from
its slot, or from the host copy with ordinary loads.  Checks:

* the output is bit-identical for an empty cache, a few slots and every
  expert in a slot, on each kernel the resident entry point runs (the
  one-token streaming kernel, the three-kernel chain, the grouped GEMV path),
  for Q2_K and Q4_K;
* on the paths it shares with ds_moe_layer (one to four tokens) it equals
  ds_moe_layer bit for bit; on the GEMV path it is within the decode
  tolerance of the fp64 oracle and the route is exact;
* the cache object (ds_moe_cache_layer) over several layers: every output
  equals ds_moe_layer, the device slot tables equal the host mirror, each
  occupied slot holds its expert's bytes, and repeated calls hit.
"""
from dataclasses import replace

import numpy as np
import pytest

import dsgen
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_quantized_routed_router_gb300 as ds  # noqa: E402
from bit_quantized_routed_router_gb300 import synthetic  # noqa: E402

DECODE_TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_routed_router_gb300 import build
    build.build()
    yield


def tiny(T, fmt="q2k", **kw):
    c = replace(dsgen.TINY, name=f"resident T={T} {fmt}", T=T, D=1024, F=1024, E=16, k=4, Fs=512,
                shared_sigma=0.02, x_dtype="bf16", router_dtype="bf16", router_sigma=0.02, seed=41,
                expert_fmt=fmt)
    return replace(c, **kw)


def pinned_copy(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def views(cfg, W, n_few, seed=0):
    """Slot tables and caches for an empty cache, n_few experts in slots and
    every expert in a slot (slots in a shuffled order)."""
    eb = ds.expert_bytes(cfg.D, cfg.F, synthetic.shape_of(cfg).expert_format)
    rng = np.random.default_rng(seed)
    per_expert = W.experts.view(cfg.E, eb)  # the packed experts, one row each
    out = []
    for n in (0, n_few, cfg.E):
        chosen = rng.permutation(cfg.E)[:n]
        slot = np.full(cfg.E, -1, np.int32)
        cache = torch.zeros((max(n, 1), eb), dtype=torch.uint8, device="cuda")
        order = rng.permutation(n)
        for s, e in zip(order, chosen):
            slot[e] = s
            cache[s].copy_(per_expert[e])
        out.append((n, torch.from_numpy(slot).cuda(), cache))
    return out


def run_resident(cfg, W, host, slot, cache, x):
    sh = synthetic.shape_of(cfg)
    T = x.shape[0]
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    out = torch.full((T, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    dbg = {"ids": torch.empty((T, cfg.k), dtype=torch.int32, device="cuda"),
           "w": torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")}
    Wr = replace(W, experts=None)
    ds.layer_resident(sh, Wr, slot, cache, host, x, out, ws, debug=dbg)
    ds.sync_status()
    return out.cpu().numpy(), dbg["ids"].cpu().numpy(), dbg["w"].cpu().numpy()


def run_layer(cfg, W, x):
    sh = synthetic.shape_of(cfg)
    T = x.shape[0]
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    out = torch.full((T, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    ds.layer(sh, W, x, out, ws)
    ds.sync_status()
    return out.cpu().numpy()


def oracle_check(cfg, x_att, out, ids, w):
    lo = oracle.LayerOracle(cfg)
    x64 = oracle.as_f64(dsgen.host_x(cfg, x_att), cfg.x_dtype)
    rids, rw = oracle.select(lo.logits(x64), cfg.k)
    assert np.array_equal(ids, rids)
    assert np.max(np.abs(w - rw)) <= 1e-5
    ref = oracle.moe_layer(x64, lo.experts(rids), lo.shared, rids, rw, cfg.D, cfg.E, cfg.F, cfg.Fs,
                           fmt=cfg.expert_fmt)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.max(np.abs(out.astype(np.float64) - ref))
    assert err <= DECODE_TOL * rms, f"max|err| {err:.3e} > {DECODE_TOL} * rms {rms:.3e}"


@pytest.mark.parametrize("T,fmt,path", [(1, "q2k", ds.PATH_STREAM), (3, "q2k", ds.PATH_DECODE3),
                                        (8, "q2k", ds.PATH_GROUPED_GEMV), (40, "q2k", ds.PATH_GROUPED_GEMV),
                                        (1, "q4k", ds.PATH_STREAM), (8, "q4k", ds.PATH_GROUPED_GEMV)])
def test_output_does_not_depend_on_the_cache(T, fmt, path):
    cfg = tiny(T, fmt)
    sh = synthetic.shape_of(cfg)
    assert ds.layer_path_resident(sh, T) == path
    lo = oracle.LayerOracle(cfg)
    att = oracle.resample_attempts(cfg, lo)
    W = synthetic.build_layer(cfg)
    x = synthetic.build_x(cfg, att)
    host = pinned_copy(W.experts)
    outs = []
    for n, slot, cache in views(cfg, W, 5, seed=T):
        out, ids, w = run_resident(cfg, W, host, slot, cache, x)
        outs.append(out)
        assert np.isfinite(out).all(), n
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    if path in (ds.PATH_STREAM, ds.PATH_DECODE3):
        assert ds.layer_path(sh, T, x) == path
        assert np.array_equal(outs[0], run_layer(cfg, W, x))
    oracle_check(cfg, att, outs[0], ids, w)


def test_flash_width_one_token_from_host_memory():
    """The Flash layer (n_embd 4096, 256 experts, top-6) for one token with
    every routed expert in host memory, and with half of them in slots:
    bit-identical to ds_moe_layer."""
    cfg = dsgen.DECODE1
    W = synthetic.build_layer(cfg)
    x = synthetic.build_x(cfg)
    host = pinned_copy(W.experts)
    ref = run_layer(cfg, W, x)
    for n, slot, cache in views(cfg, W, cfg.E // 2, seed=3)[:2]:
        out, _, _ = run_resident(cfg, W, host, slot, cache, x)
        assert np.array_equal(out, ref), n


@pytest.mark.parametrize("n_slots", [0, 6, 48])
def test_cache_object_over_layers(n_slots):
    n_layers = 3
    cfg = tiny(1)
    sh = synthetic.shape_of(cfg)
    Ws = [synthetic.build_layer(cfg, layer=l) for l in range(n_layers)]
    hosts = [pinned_copy(W.experts) for W in Ws]
    eb = ds.expert_bytes(cfg.D, cfg.F, sh.expert_format)
    slots = torch.zeros((max(n_slots, 1), eb), dtype=torch.uint8, device="cuda")
    tables = torch.zeros((n_layers, cfg.E), dtype=torch.int32, device="cuda")
    c = ds.ExpertCache(sh, hosts, slots, n_slots, tables)
    ws = torch.empty(ds.workspace_bytes(sh, 2), dtype=torch.uint8, device="cuda")
    try:
        for rep in range(3):
            for l in range(n_layers):
                T = 1 + (rep + l) % 2  # the streaming kernel and the chain
                x = synthetic.build_x(cfg, layer=l + 10 * (rep % 2), T=T)
                out = torch.full((T, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
                c.layer(l, replace(Ws[l], experts=None), x, out, ws)
                ds.sync_status()
                assert np.array_equal(out.cpu().numpy(), run_layer(cfg, Ws[l], x)), (rep, l)
        tab = tables.cpu().numpy()
        for l in range(n_layers):
            for e in range(cfg.E):
                s = c.slot(l, e)
                assert tab[l, e] == s
                if s >= 0:
                    assert torch.equal(slots[s], Ws[l].experts.view(cfg.E, eb)[e])
        st = c.stats()
        assert st["resident"] == min(n_slots, st["misses"])
        if n_slots >= n_layers * cfg.E:
            assert st["hits"] > 0
        if n_slots == 0:
            assert st["hits"] == 0
    finally:
        c.close()


def test_zero_tokens_and_cache_gemv_path():
    """T = 0 through the resident entry point and the cache object is a
    no-op; an eight-token call through the cache (the GEMV path) matches the
    oracle and fills slots like any other call."""
    cfg = tiny(8)
    sh = synthetic.shape_of(cfg)
    W = synthetic.build_layer(cfg)
    host = pinned_copy(W.experts)
    eb = ds.expert_bytes(cfg.D, cfg.F, sh.expert_format)
    slot = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(ds.workspace_bytes(sh, 8), dtype=torch.uint8, device="cuda")
    x0 = torch.empty((0, cfg.D), dtype=torch.int16, device="cuda")
    out0 = torch.empty((0, cfg.D), dtype=torch.float32, device="cuda")
    ds.layer_resident(sh, replace(W, experts=None), slot, None, host, x0, out0, ws)
    slots = torch.zeros((4, eb), dtype=torch.uint8, device="cuda")
    tables = torch.zeros((1, cfg.E), dtype=torch.int32, device="cuda")
    c = ds.ExpertCache(sh, [host], slots, 4, tables)
    try:
        c.layer(0, replace(W, experts=None), x0, out0, ws)
        assert c.stats() == {"hits": 0, "misses": 0, "resident": 0}
        lo = oracle.LayerOracle(cfg)
        att = oracle.resample_attempts(cfg, lo)
        x = synthetic.build_x(cfg, att)
        out = torch.full((8, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
        c.layer(0, replace(W, experts=None), x, out, ws)
        ds.sync_status()
        assert c.stats()["resident"] == 4
        lo_x = oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype)
        rids, rw = oracle.select(lo.logits(lo_x), cfg.k)
        ref = oracle.moe_layer(lo_x, lo.experts(rids), lo.shared, rids, rw, cfg.D, cfg.E, cfg.F, cfg.Fs,
                               fmt=cfg.expert_fmt)
        got = out.cpu().numpy().astype(np.float64)
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.max(np.abs(got - ref)) <= DECODE_TOL * rms
    finally:
        c.close()

