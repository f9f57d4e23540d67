"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bit-exact: Q2_K bytes, dequantised weights, expert ids (and their order),
per-expert counts, offsets and the permutation.  Floats: max|err| <= tol *
rms(out_oracle) with tol = 2e-3 on the decode path and 5e-3 on the
prefill path; the oracle's routing weights and logits are compared at the
same scale.  Tokens are resampled (oracle-side) until no two of their top
k+1 logits lie within 1e-4, so the selection has one answer at fp32.
"""
import numpy as np
import pytest

import dsgen
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_quantized_routed_router_gb300 as ds  # noqa: E402
from bit_quantized_routed_router_gb300 import synthetic  # noqa: E402

DECODE_TOL = 2e-3
PREFILL_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_routed_router_gb300 import build
    build.build()
    yield


def gpu_quantize(w_np):
    w = torch.from_numpy(np.ascontiguousarray(w_np, np.float32)).cuda()
    out = torch.zeros(ds.q2k_bytes(*w.shape), dtype=torch.uint8, device="cuda")
    ds.quantize_q2k(w, out)
    ds.sync_status()
    return out.cpu().numpy().reshape(w.shape[0], -1)


def run_layer(cfg, W, x, scale=1.0, logit_scale=1.0, bias_select_only=0):
    T = x.shape[0]
    sh = synthetic.shape_of(cfg)
    sh.routed_scale = scale
    sh.logit_scale = logit_scale
    sh.bias_select_only = bias_select_only
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, cfg.D), dtype=torch.float32, device="cuda")
    P = T * cfg.k
    dbg = {"logits": torch.empty((T, cfg.E), dtype=torch.float32, device="cuda"),
           "ids": torch.empty((T, cfg.k), dtype=torch.int32, device="cuda"),
           "w": torch.empty((T, cfg.k), dtype=torch.float32, device="cuda"),
           "counts": torch.empty(cfg.E, dtype=torch.int32, device="cuda"),
           "offsets": torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda"),
           "perm": torch.empty(P, dtype=torch.int32, device="cuda")}
    ds.layer(sh, W, x, out, ws, debug=dbg)
    ds.sync_status()
    return out.cpu().numpy(), {k: v.cpu().numpy() for k, v in dbg.items()}


def check_route(dbg, ids_ref, E, rows=None):
    """ids (and order) for the given rows; counts/offsets/perm over the batch."""
    ids = dbg["ids"] if rows is None else dbg["ids"][rows]
    assert np.array_equal(ids, ids_ref)


def check_route_full(dbg, ids_ref, E):
    assert np.array_equal(dbg["ids"], ids_ref)
    counts, offsets, perm, _ = oracle.route(ids_ref, E)
    assert np.array_equal(dbg["counts"], counts)
    assert np.array_equal(dbg["offsets"], offsets)
    assert np.array_equal(dbg["perm"], perm)


def check_close(got, ref, tol, what="out"):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.max(np.abs(got.astype(np.float64) - ref))
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e}"
    print(f"{what}: max|err|/rms = {err / rms:.3e}")
    return err / rms


# ------------------------------------------------------------- quantiser --

@pytest.mark.parametrize("rows,in_dim,scale", [(3, 256, 0.02), (5, 128, 1.0), (4, 300, 5.0),
                                               (64, 1024, 0.02), (2, 256, 1e4), (2, 512, 1e-30)])
def test_quantize_bit_exact_random(rows, in_dim, scale):
    rng = np.random.default_rng(rows * 1000 + in_dim)
    x = (rng.normal(size=(rows, in_dim)) * scale).astype(np.float32)
    x[0, :16] = np.abs(x[0, :16])
    if rows > 1:
        x[1, 16:32] = 0.0
        x[1, 32:48] = -np.abs(x[1, 32:48])
    assert np.array_equal(gpu_quantize(x), oracle.quantize(x))


def test_quantize_domain_edges():
    x = np.zeros((3, 256), np.float32)
    x[0, 0], x[0, 1] = 65504.0, -65504.0
    x[1, 7] = 1e-45   # fp32 subnormal
    x[2, :] = np.linspace(-3.0, 7.0, 256)
    assert np.array_equal(gpu_quantize(x), oracle.quantize(x))
    bad = np.zeros((1, 256), np.float32)
    bad[0, 9] = 65505.0
    with pytest.raises(ValueError):
        oracle.quantize(bad)
    with pytest.raises(ds.DsMoeError):
        gpu_quantize(bad)


def test_quantize_bit_exact_generated_expert():
    cfg = dsgen.DECODE1
    g, u, d = dsgen.host_expert_f32(cfg, 17)
    for m in (g, d):
        assert np.array_equal(gpu_quantize(m), oracle.quantize(m))


def test_quantize_nonfinite_sets_status():
    x = np.zeros((2, 256), np.float32)
    x[1, 5] = np.inf
    w = torch.from_numpy(x).cuda()
    out = torch.full((ds.q2k_bytes(2, 256),), 7, dtype=torch.uint8, device="cuda")
    ds.quantize_q2k(w, out)
    with pytest.raises(ds.DsMoeError) as ei:
        ds.sync_status()
    assert ei.value.code == ds.DS_ERR_DEVICE_CHECK
    o = out.cpu().numpy()
    assert not o[84:].any()          # the bad block is zeroed
    assert np.array_equal(o[:84], oracle.quantize(x[:1]).ravel())
    ds.sync_status()                 # the status word was cleared


def test_dequantize_bit_exact():
    rng = np.random.default_rng(3)
    x = (rng.normal(size=(16, 512)) * 0.02).astype(np.float32)
    q = oracle.quantize(x)
    blocks = rng.integers(0, 256, (4, 3 * 84)).astype(np.uint8)
    for r in range(4):
        for b in range(3):
            for o in (80, 82):  # finite d and dmin, some subnormal
                v = int(rng.integers(0, 0x7BFF))
                blocks[r, 84 * b + o], blocks[r, 84 * b + o + 1] = v & 0xFF, v >> 8
    for qq, rows, in_dim in ((q, 16, 512), (blocks, 4, 700)):
        ref = oracle.dequantize(qq, rows, in_dim).astype(np.float32)  # fp32 of the exact value
        out = torch.empty((rows, in_dim), dtype=torch.float32, device="cuda")
        ds.dequantize_q2k(torch.from_numpy(qq).cuda(), rows, in_dim, out)
        ds.sync_status()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ----------------------------------------------------------------- layers --

def oracle_case(cfg, layer=0):
    lo = oracle.LayerOracle(cfg, layer)
    att = oracle.resample_attempts(cfg, lo)
    x = oracle.as_f64(dsgen.host_x(cfg, att, layer), cfg.x_dtype)
    return lo, att, x


def layer_parity(cfg, tol, scale=1.0, logit_scale=1.0, bias_select_only=0, W=None):
    lo, att, x64 = oracle_case(cfg)
    W = synthetic.build_layer(cfg) if W is None else W
    x = synthetic.build_x(cfg, att)
    out, dbg = run_layer(cfg, W, x, scale, logit_scale, bias_select_only)
    L = lo.logits(x64)
    ids, w = oracle.select(L, cfg.k, scale, logit_scale, lo.bias if bias_select_only else None)
    check_route_full(dbg, ids, cfg.E)
    res = oracle.moe_layer(x64, lo.experts(ids), lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs,
                           fmt=cfg.expert_fmt)
    check_close(dbg["logits"], L, 1e-5, "logits")
    assert np.max(np.abs(dbg["w"] - w)) <= 1e-5
    return check_close(out, res, tol)


def test_tiny_layer_parity():
    layer_parity(dsgen.TINY, DECODE_TOL)


@pytest.mark.parametrize("variant", ["k_eq_E", "one_expert", "shared", "scale1.5", "logit1.5", "T33",
                                     "T1", "T2logit1.5", "zipf", "zipf_select_only"])
def test_tiny_variants(variant):
    """Variants of the tiny layer; logit1.5 scales the selected logits before
    the softmax (the grouped path's selection kernel; T2logit1.5: the
    three-kernel path's router warp)."""
    from dataclasses import replace
    c = dsgen.TINY
    scale = 1.0
    logit_scale = 1.0
    if variant == "k_eq_E":
        c = replace(c, k=16)
    elif variant == "one_expert":
        c = replace(c, E=1, k=1)
    elif variant == "shared":
        c = replace(c, Fs=128, shared_sigma=0.02)
    elif variant == "scale1.5":
        scale = 1.5
    elif variant == "logit1.5":
        logit_scale = 1.5
    elif variant == "T2logit1.5":
        c = replace(c, T=2)
        logit_scale = 1.5
    elif variant in ("zipf", "zipf_select_only"):
        c = replace(c, zipf_s=1.1)
        if variant == "zipf_select_only":
            layer_parity(c, DECODE_TOL, bias_select_only=1)
            return
    elif variant == "T33":
        c = replace(c, T=33, k=3)
    elif variant == "T1":
        c = replace(c, T=1)
    layer_parity(c, DECODE_TOL, scale, logit_scale)


def _small(T, Fs, k=2, E=16, dtype="f32"):
    from dataclasses import replace
    return replace(dsgen.TINY, name=f"small D=1024 F=1024 T={T} Fs={Fs} k={k} E={E} {dtype}", T=T,
                   D=1024, F=1024, E=E, k=k, Fs=Fs, shared_sigma=0.02, x_dtype=dtype,
                   router_dtype=dtype)


@pytest.mark.parametrize("T,Fs,k,E,dtype", [(1, 0, 2, 16, "f32"), (2, 256, 2, 16, "f32"),
                                            (1, 512, 6, 16, "bf16"), (1, 0, 16, 16, "f32"),
                                            (2, 1024, 4, 40, "bf16"), (1, 128, 1, 3, "f32"),
                                            (3, 256, 2, 16, "f32"), (4, 256, 4, 16, "f32"),
                                            (1, 512, 8, 16, "bf16"), (8, 0, 16, 16, "f32")])
def test_small_decode_variants(T, Fs, k, E, dtype):
    """Decode-sized batches at a reduced width: the one-token kernel (up to its
    largest top-k, 8), the three-kernel chain (up to four tokens here: fp32
    inputs do not take the batched kernels) and the grouped path, including
    k = E, one expert per token, odd E and no shared expert."""
    layer_parity(_small(T, Fs, k, E, dtype), DECODE_TOL)


def test_tiny_prefill_sized_batch():
    """A batch beyond the decode size takes the large-batch route kernels and,
    with fp32 inputs, the grouped GEMV path (fp32 arithmetic): decode
    tolerance."""
    from dataclasses import replace
    c = replace(dsgen.TINY, T=700, k=2)
    assert ds.layer_path(synthetic.shape_of(c), c.T) == ds.PATH_GROUPED_GEMV
    layer_parity(c, DECODE_TOL)


def _tc(T, Fs, k, E, zipf=0.0, seed=7):
    from dataclasses import replace
    return replace(dsgen.TINY, name=f"tc D=1024 F=1024 T={T} Fs={Fs} k={k} E={E} zipf={zipf}", T=T,
                   D=1024, F=1024, E=E, k=k, Fs=Fs, shared_sigma=0.02, x_dtype="bf16",
                   router_dtype="bf16", router_sigma=0.02, zipf_s=zipf, seed=seed)


def wide_layout(counts):
    """Whether the tile plan takes token chunks of up to 256 (Q2_K): when they
    cut the routed chunks of up to 128 by more than a tenth."""
    used = counts[counts > 0]
    n128, n256 = int(np.sum((used + 127) // 128)), int(np.sum((used + 255) // 256))
    return 10 * n256 < 9 * n128


@pytest.mark.parametrize("T,Fs,k,E,zipf,wide", [(300, 1024, 4, 16, 0.0, False), (64, 1024, 2, 8, 0.0, False),
                                                 (200, 0, 6, 40, 0.0, False), (520, 1024, 6, 32, 1.1, True),
                                                 (600, 1024, 6, 8, 0.0, True)])
def test_prefill_tensor_core_path(T, Fs, k, E, zipf, wide):
    """Batches of 64 tokens or more with bf16 inputs and widths that are
    multiples of 1024 run the expert FFNs as grouped tcgen05 GEMMs: the whole
    output against the oracle at the prefill tolerance.  The cases cover the
    smallest batch of the path, several 128-token chunks per expert (ragged
    last chunks), no shared expert, an odd expert count, and, in the wide
    layout (tiles of up to 256 tokens), a Zipf-skewed route whose hottest
    experts exceed one 256-token chunk and a route of about 450 tokens per
    expert (ragged 256-token chunks)."""
    cfg = _tc(T, Fs, k, E, zipf)
    assert ds.layer_path(synthetic.shape_of(cfg), T) == ds.PATH_TENSOR_CORE
    lo, att, x64 = oracle_case(cfg)
    ids, _ = oracle.select(lo.logits(x64), cfg.k)
    assert wide_layout(np.bincount(ids.ravel(), minlength=cfg.E)) == wide
    layer_parity(cfg, PREFILL_TOL)


def test_layer_path_selection():
    """The kernels each decode and prefill workload runs on."""
    from dataclasses import replace
    sh = synthetic.shape_of(dsgen.DECODE1)
    assert ds.layer_path(sh, 0) == ds.PATH_NONE
    assert ds.layer_path(sh, 1) == ds.PATH_STREAM
    assert ds.layer_path(sh, 3) == ds.PATH_DECODE3
    assert ds.layer_path(sh, 4) == ds.PATH_BATCHED_DECODE
    assert ds.layer_path(sh, 5) == ds.PATH_BATCHED_DECODE
    assert ds.layer_path(sh, 8) == ds.PATH_BATCHED_DECODE
    assert ds.layer_path(sh, 16) == ds.PATH_BATCHED_DECODE
    assert ds.layer_path(sh, 17) == ds.PATH_TENSOR_CORE
    assert ds.layer_path(sh, 32) == ds.PATH_TENSOR_CORE
    assert ds.layer_path(synthetic.shape_of(dsgen.PREFILL), 4096) == ds.PATH_TENSOR_CORE
    assert ds.layer_path(synthetic.shape_of(dsgen.TINY), 700) == ds.PATH_GROUPED_GEMV  # fp32 x
    assert ds.layer_path(synthetic.shape_of(replace(dsgen.DECODE1, T=1)), 64) == ds.PATH_TENSOR_CORE


@pytest.fixture(scope="module")
def decode1():
    cfg = dsgen.DECODE1
    lo, att, x64 = oracle_case(cfg)
    return cfg, lo, att, x64, synthetic.build_layer(cfg)


def test_decode_b1_parity(decode1):
    cfg, lo, att, x64, W = decode1
    out, dbg = run_layer(cfg, W, synthetic.build_x(cfg, att))
    (res, ids, w, L) = lo.forward(x64)
    check_route_full(dbg, ids, cfg.E)
    check_close(dbg["logits"], L, 1e-5, "logits")
    check_close(out, res, DECODE_TOL)


def test_decode_b1_logit_scale(decode1):
    """Flash decode B=1 (the one-token kernel's router warp) with both
    readings of the pages' 1.5: weights scaled, and logits scaled before the
    softmax."""
    cfg, lo, att, x64, W = decode1
    out, dbg = run_layer(cfg, W, synthetic.build_x(cfg, att), 1.5, 1.5)
    L = lo.logits(x64)
    ids, w = oracle.select(L, cfg.k, 1.5, 1.5)
    check_route_full(dbg, ids, cfg.E)
    assert np.max(np.abs(dbg["w"] - w)) <= 1e-5
    res = oracle.moe_layer(x64, lo.experts(ids), lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs,
                           fmt=cfg.expert_fmt)
    check_close(out, res, DECODE_TOL)


def test_zipf_bias_for_selection_only_decode_paths():
    """The Flash layer with the Zipf router bias steering the selection only,
    on the one-token kernel (T=1), the three-kernel chain (T=3) and the
    batched decode path (T=8): weights from the unbiased selected logits."""
    from dataclasses import replace
    W = synthetic.build_layer(dsgen.DECODE32_ZIPF)
    for T in (1, 3, 8):
        layer_parity(replace(dsgen.DECODE32_ZIPF, T=T), DECODE_TOL, bias_select_only=1, W=W)


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_hostio_matches_device(decode1, pinned):
    """The host-buffer entry point gives the device path's output bit for bit:
    with pinned buffers the kernels read x and write out in host memory
    directly; with pageable ones the library copies around the layer."""
    cfg, lo, att, x64, W = decode1
    x = synthetic.build_x(cfg, att)
    out_dev, _ = run_layer(cfg, W, x)
    sh = synthetic.shape_of(cfg)
    ws = torch.empty(ds.workspace_bytes(sh, 1), dtype=torch.uint8, device="cuda")
    xh = x.cpu()
    oh = torch.full((1, cfg.D), float("nan"), dtype=torch.float32)
    if pinned:
        xh, oh = xh.pin_memory(), oh.pin_memory()
    for _ in range(2):  # the second call reuses the workspace's staged copy region
        ds.layer_hostio(sh, W, xh, oh, ws)
        ds.sync_status()
        assert np.array_equal(oh.numpy(), out_dev)


def test_decode32_zipf_parity():
    cfg = dsgen.DECODE32_ZIPF
    layer_parity(cfg, DECODE_TOL)


def test_batch_invariance_decode(decode1):
    """Within one path a token's result does not depend on its batch: tokens of
    an 8-token batch equal the same tokens in 5- and 4-token batches bit for
    bit (batched decode path), and tokens of a 2-token batch equal the same
    tokens in a 3-token batch (three-kernel path).  A token alone takes the
    one-token streaming kernel; every path agrees with the others at
    tolerance."""
    cfg, lo, att, x64, W = decode1
    from dataclasses import replace
    c8 = replace(cfg, T=8)
    xb = synthetic.build_x(c8)
    out_b, _ = run_layer(c8, W, xb)
    out_5, _ = run_layer(replace(cfg, T=5), W, xb[2:7].contiguous())
    assert np.array_equal(out_5, out_b[2:7])
    out_4, _ = run_layer(replace(cfg, T=4), W, xb[4:8].contiguous())
    assert np.array_equal(out_4, out_b[4:8])
    out_3, _ = run_layer(replace(cfg, T=3), W, xb[0:3].contiguous())
    out_2, _ = run_layer(replace(cfg, T=2), W, xb[0:2].contiguous())
    assert np.array_equal(out_2, out_3[0:2])
    for t in (0, 2):
        out_1, _ = run_layer(cfg, W, xb[t:t + 1].contiguous())
        check_close(out_1[0].astype(np.float64), out_3[t].astype(np.float64), DECODE_TOL,
                    "one-token kernel vs three-kernel path")
        check_close(out_1[0].astype(np.float64), out_b[t].astype(np.float64), DECODE_TOL,
                    "one-token kernel vs batched decode path")


@pytest.mark.parametrize("T", [1, 3])
def test_back_to_back_layers_read_the_previous_output(T):
    """Layers enqueued back to back, each reading the previous layer's output
    as its x (fp32 x and router, so that out feeds x directly): the router
    grid of a layer may launch while the previous layer's kernels still run,
    and must read x only after they have completed.  The outputs equal those
    of the same calls with the stream synchronised between layers, bit for
    bit, both eagerly and replayed from a CUDA graph."""
    from dataclasses import replace
    cfg = replace(dsgen.DECODE1, T=T, x_dtype="f32", router_dtype="f32", name=f"chain of layers T={T}")
    sh = synthetic.shape_of(cfg)
    assert ds.layer_path(sh, T) == (ds.PATH_STREAM if T == 1 else ds.PATH_DECODE3)
    Ws = [synthetic.build_layer(cfg, layer=l) for l in range(4)]
    x0 = synthetic.build_x(cfg)
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    bufs = [torch.empty((T, cfg.D), dtype=torch.float32, device="cuda") for _ in range(4)]

    def run(sync):
        x = x0
        for l in range(4):
            ds.layer(sh, Ws[l], x, bufs[l], ws)
            if sync:
                torch.cuda.synchronize()
            x = bufs[l]

    run(True)
    ref = [b.cpu().numpy().copy() for b in bufs]
    assert all(np.isfinite(r).all() for r in ref)
    for b in bufs:
        b.fill_(float("nan"))
    for _ in range(3):
        run(False)
    torch.cuda.synchronize()
    ds.sync_status()
    for l in range(4):
        assert np.array_equal(bufs[l].cpu().numpy(), ref[l]), f"layer {l}"
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(False)
    for b in bufs:
        b.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ds.sync_status()
    for l in range(4):
        assert np.array_equal(bufs[l].cpu().numpy(), ref[l]), f"layer {l} (graph)"


def test_batch_invariance_small_width():
    """At width 1024: tokens of a 2-token batch equal the same tokens in a
    3-token batch bit for bit (three-kernel path); a token alone (one-token
    streaming kernel) agrees with them at tolerance, and is deterministic."""
    cfg = _small(3, 256, 2, 16, "bf16")
    from dataclasses import replace
    W = synthetic.build_layer(cfg)
    xb = synthetic.build_x(cfg)
    out_3, _ = run_layer(cfg, W, xb)
    out_2, _ = run_layer(replace(cfg, T=2), W, xb[0:2].contiguous())
    assert np.array_equal(out_2, out_3[0:2])
    for t in (0, 2):
        out_1, _ = run_layer(replace(cfg, T=1), W, xb[t:t + 1].contiguous())
        again, _ = run_layer(replace(cfg, T=1), W, xb[t:t + 1].contiguous())
        assert np.array_equal(out_1, again)
        check_close(out_1[0].astype(np.float64), out_3[t].astype(np.float64), DECODE_TOL,
                    "one-token kernel vs three-kernel path")


@pytest.mark.parametrize("cfg", [dsgen.PREFILL, dsgen.PREFILL_ZIPF], ids=["uniform", "zipf"])
def test_prefill_parity_full(cfg):
    """Flash prefill, T = 4096, on the tensor cores: every row of the output
    against the oracle (all 256 experts dequantised once each), with the
    uniform router (about 96 tokens per expert) and the Zipf-skewed one (the
    hottest experts serve thousands of tokens in many 128-token chunks)."""
    lo = oracle.LayerOracle(cfg)
    att = oracle.resample_attempts(cfg, lo)
    W = synthetic.build_layer(cfg)
    assert ds.layer_path(synthetic.shape_of(cfg), cfg.T) == ds.PATH_TENSOR_CORE
    out, dbg = run_layer(cfg, W, synthetic.build_x(cfg, att))
    del W
    torch.cuda.empty_cache()
    x64 = oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype)
    L = lo.logits(x64)
    ids, w = oracle.select(L, cfg.k)
    check_route_full(dbg, ids, cfg.E)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    print(f"{cfg.name}: {int((counts > 0).sum())} experts used, hottest {int(counts.max())} tokens")
    res = oracle.moe_layer(x64, lo.experts(ids), lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs,
                           fmt=cfg.expert_fmt)
    check_close(out, res, PREFILL_TOL)


def test_zero_tokens_is_noop(decode1):
    cfg, lo, att, x64, W = decode1
    sh = synthetic.shape_of(cfg)
    out = torch.full((1, cfg.D), 3.0, device="cuda")
    ws = torch.empty(ds.workspace_bytes(sh, 1), dtype=torch.uint8, device="cuda")
    ds.layer(sh, W, synthetic.build_x(cfg, att), out, ws, T=0)
    ds.sync_status()
    assert torch.all(out == 3.0)


def test_stack_parity_by_layer():
    """The stack  x <- x + layer(bf16(RMSNorm(x)))  at full width, T=8, all
    43 layers, at the decode tolerance (a batch of 8 runs the batched decode
    path).  Every layer is checked on the residual the GPU itself produced
    before it: the oracle normalises that residual, runs the layer in fp64 and
    adds it, and the GPU's next residual must match within 2e-3 * rms of the
    update.  Comparing whole trajectories instead would not test the kernels:
    routing is discontinuous, and residual differences at the level of the
    float tolerance move logits by far more than the 1e-4 gap the generator
    guarantees, so after a few layers a token may rightly take another expert
    on one side.  A token whose logits on the GPU's residual have a near-tie
    (gap < 1e-4) is left out of that layer's comparison.  ds_moe_stack over
    several layers is bit-identical to these one-layer calls (next test)."""
    from dataclasses import replace
    cfg = dsgen.STACK
    sh = synthetic.shape_of(cfg)
    assert ds.layer_path(sh, cfg.T) == ds.PATH_BATCHED_DECODE
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(dsgen.host_x(replace(cfg, x_dtype="f32"))).cuda()
    checked, worst = 0, 0.0
    for l in range(cfg.layers):
        W = synthetic.build_layer(cfg, l)
        x_in = x.cpu().numpy()
        ds.stack(sh, [W], x, ws)
        ds.sync_status()
        del W
        got = x.cpu().numpy().astype(np.float64) - x_in
        lo = oracle.LayerOracle(cfg, l)
        r64 = oracle.as_f64(oracle.rmsnorm_bf16(x_in), "bf16")
        res, _, _, L = lo.forward(r64)
        keep = oracle.min_top_gap(L, cfg.k) >= oracle.GAP
        ref = (x_in.astype(np.float64) + res).astype(np.float32).astype(np.float64) - x_in
        r = check_close(got[keep], ref[keep], DECODE_TOL, f"stack layer {l} ({keep.sum()} tokens)")
        worst = max(worst, r)
        checked += int(keep.sum())
    print(f"stack: {cfg.layers} layers, {checked} token-layers checked, worst max|err|/rms = {worst:.2e}")
    assert checked >= cfg.layers * cfg.T - 8


def test_stack_equals_layer_by_layer():
    """ds_moe_stack is bit-identical to RMSNorm + ds_moe_layer + residual add
    issued one layer at a time (here 4 layers)."""
    from dataclasses import replace
    cfg = dsgen.STACK
    Ws = [synthetic.build_layer(cfg, l) for l in range(4)]
    sh = synthetic.shape_of(cfg)
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device="cuda")
    x0 = torch.from_numpy(dsgen.host_x(replace(cfg, x_dtype="f32"))).cuda()
    xa = x0.clone()
    ds.stack(sh, Ws, xa, ws)
    xb = x0.clone()
    for W in Ws:
        xb_in = xb.clone()
        ds.stack(sh, [W], xb, ws)
        assert not torch.equal(xb, xb_in)
    ds.sync_status()
    assert torch.equal(xa, xb)


# ------------------------------------------------------------------ Q4_K --
# The 144-byte Q4_K experts ("Understanding Dwarf Star", 2.3.2): quantiser
# and dequantiser bit-exact, the layer at the decode tolerance (the grouped
# dequantising GEMV path with fp32 arithmetic serves every batch size).

def gpu_quantize_q4k(w_np):
    w = torch.from_numpy(np.ascontiguousarray(w_np, np.float32)).cuda()
    out = torch.zeros(ds.q4k_bytes(*w.shape), dtype=torch.uint8, device="cuda")
    ds.quantize_q4k(w, out)
    ds.sync_status()
    return out.cpu().numpy().reshape(w.shape[0], -1)


@pytest.mark.parametrize("rows,in_dim,scale", [(3, 256, 0.02), (5, 128, 1.0), (4, 300, 5.0),
                                               (64, 1024, 0.02), (2, 256, 1e4), (2, 512, 1e-30)])
def test_q4k_quantize_bit_exact_random(rows, in_dim, scale):
    rng = np.random.default_rng(rows * 1000 + in_dim + 1)
    x = (rng.normal(size=(rows, in_dim)) * scale).astype(np.float32)
    x[0, :32] = np.abs(x[0, :32])
    if rows > 1:
        x[1, 32:64] = 0.0
        x[1, 64:96] = -np.abs(x[1, 64:96])
    assert np.array_equal(gpu_quantize_q4k(x), oracle.quantize_q4k(x))


def test_q4k_quantize_domain_edges_and_status():
    x = np.zeros((3, 256), np.float32)
    x[0, 0], x[0, 1] = 65504.0, -65504.0
    x[1, 7] = 1e-45
    x[2, :] = np.linspace(-3.0, 7.0, 256)
    assert np.array_equal(gpu_quantize_q4k(x), oracle.quantize_q4k(x))
    g, _, d = dsgen.host_expert_f32(dsgen.DECODE1, 17)
    assert np.array_equal(gpu_quantize_q4k(d), oracle.quantize_q4k(d))
    bad = np.zeros((2, 256), np.float32)
    bad[1, 5] = np.nan
    w = torch.from_numpy(bad).cuda()
    out = torch.full((ds.q4k_bytes(2, 256),), 7, dtype=torch.uint8, device="cuda")
    ds.quantize_q4k(w, out)
    with pytest.raises(ds.DsMoeError) as ei:
        ds.sync_status()
    assert ei.value.code == ds.DS_ERR_DEVICE_CHECK
    o = out.cpu().numpy()
    assert not o[144:].any() and not o[:144].any()   # bad block zeroed; the zero block is all zero
    ds.sync_status()


def test_q4k_dequantize_bit_exact():
    rng = np.random.default_rng(4)
    x = (rng.normal(size=(16, 512)) * 0.02).astype(np.float32)
    q = oracle.quantize_q4k(x)
    blocks = rng.integers(0, 256, (4, 3 * 144)).astype(np.uint8)
    for r in range(4):
        for b in range(3):
            for o in (0, 2):
                v = int(rng.integers(0, 0x7BFF))
                blocks[r, 144 * b + o], blocks[r, 144 * b + o + 1] = v & 0xFF, v >> 8
    for qq, rows, in_dim in ((q, 16, 512), (blocks, 4, 700)):
        ref = oracle.dequantize_q4k(qq, rows, in_dim).astype(np.float32)
        out = torch.empty((rows, in_dim), dtype=torch.float32, device="cuda")
        ds.dequantize_q4k(torch.from_numpy(qq).cuda(), rows, in_dim, out)
        ds.sync_status()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("T,Fs,k,E,dtype,D", [(8, 0, 2, 16, "f32", 1024), (1, 512, 6, 16, "bf16", 1024),
                                              (1, 0, 8, 16, "f32", 1024), (1, 256, 2, 16, "f32", 512),
                                              (3, 256, 2, 16, "f32", 1024), (2, 512, 6, 16, "bf16", 1024),
                                              (4, 256, 4, 40, "f32", 1024), (33, 1024, 4, 40, "bf16", 1024)])
def test_q4k_layer_parity(T, Fs, k, E, dtype, D):
    """Q4_K experts on every decode-sized path: one token at the instantiated
    widths runs the streaming kernel, two to four tokens the three-kernel
    chain (integer dots on 4-bit codes), fp32 inputs beyond that the grouped
    GEMV path and bf16 inputs of five tokens or more the tensor cores."""
    from dataclasses import replace
    cfg = replace(_small(T, Fs, k, E, dtype), expert_fmt="q4k", D=D, F=D)
    sh = synthetic.shape_of(cfg)
    if D == 1024 and T == 1:
        path = ds.PATH_STREAM
    elif D == 1024 and T <= 4:
        path = ds.PATH_DECODE3
    elif dtype == "bf16" and T >= 5:
        path = ds.PATH_TENSOR_CORE
    else:
        path = ds.PATH_GROUPED_GEMV
    assert ds.layer_path(sh, T) == path
    layer_parity(cfg, DECODE_TOL)


@pytest.mark.parametrize("T,Fs,k,E,zipf", [(64, 1024, 2, 8, 0.0), (300, 1024, 4, 16, 0.0),
                                            (520, 1024, 6, 32, 1.1), (200, 0, 6, 40, 0.0)])
def test_q4k_tensor_core_path(T, Fs, k, E, zipf):
    """Q4_K experts on the tensor cores (the 144-byte blocks copied whole,
    dequantised to fp16 by the dequant warps): the whole output against the
    oracle at the prefill tolerance, including several 128-token chunks per
    expert, a Zipf route and no shared expert."""
    from dataclasses import replace
    cfg = replace(_tc(T, Fs, k, E, zipf, seed=9), expert_fmt="q4k")
    assert ds.layer_path(synthetic.shape_of(cfg), T) == ds.PATH_TENSOR_CORE
    layer_parity(cfg, PREFILL_TOL)


def test_q4k_decode_sized_tensor_core_batch():
    """A decode-sized Q4_K batch beyond the three-kernel chain with bf16
    inputs (17 tokens at the Flash widths) on the tensor cores, at the decode
    tolerance."""
    from dataclasses import replace
    cfg = replace(dsgen.DECODE1, T=17, expert_fmt="q4k")
    assert ds.layer_path(synthetic.shape_of(cfg), cfg.T) == ds.PATH_TENSOR_CORE
    layer_parity(cfg, DECODE_TOL)


@pytest.mark.parametrize("variant", ["one_expert", "k_eq_E", "zipf_select_only", "T1_zipf"])
def test_q4k_tiny_variants(variant):
    """Degenerate and biased routings with Q4_K experts: one expert (k = 1),
    every expert selected (k = E), a Zipf router bias that steers the
    selection only, and one token with a Zipf bias (the streaming kernel at
    width 1024)."""
    from dataclasses import replace
    c = replace(dsgen.TINY, expert_fmt="q4k")
    if variant == "one_expert":
        layer_parity(replace(c, E=1, k=1), DECODE_TOL)
    elif variant == "k_eq_E":
        layer_parity(replace(c, k=16), DECODE_TOL)
    elif variant == "zipf_select_only":
        layer_parity(replace(c, zipf_s=1.1), DECODE_TOL, bias_select_only=1)
    else:
        cfg = replace(_small(1, 512, 6, 64, "bf16"), expert_fmt="q4k", zipf_s=1.1)
        assert ds.layer_path(synthetic.shape_of(cfg), 1) == ds.PATH_STREAM
        layer_parity(cfg, DECODE_TOL)


def test_q4k_tiny_ragged_width():
    """n_ff = 128: half a Q4_K block per down row (zero-padded sub-blocks)."""
    from dataclasses import replace
    layer_parity(replace(dsgen.TINY, expert_fmt="q4k"), DECODE_TOL)


@pytest.fixture(scope="module")
def decode1_q4k():
    from dataclasses import replace
    cfg = replace(dsgen.DECODE1, expert_fmt="q4k")
    return cfg, synthetic.build_layer(cfg)


def test_q4k_decode_b1_flash_shape(decode1_q4k):
    cfg, W = decode1_q4k
    assert ds.expert_bytes(cfg.D, cfg.F, ds.DS_Q4_K) == cfg.expert_bytes == 3 * 2048 * 16 * 144
    assert ds.layer_path(synthetic.shape_of(cfg), 1) == ds.PATH_STREAM
    layer_parity(cfg, DECODE_TOL, W=W)


def test_q4k_decode_b1_hostio_and_gemv_agree(decode1_q4k):
    """The one-token Q4_K layer from pinned host buffers equals the device
    call bit for bit; the three-kernel chain (a two-token batch of the same
    token twice) agrees within the decode tolerance."""
    cfg, W = decode1_q4k
    lo, att, x64 = oracle_case(cfg)
    sh = synthetic.shape_of(cfg)
    x = synthetic.build_x(cfg, att)
    ws = torch.empty(ds.workspace_bytes(sh, 2), dtype=torch.uint8, device="cuda")
    out = torch.empty((1, cfg.D), dtype=torch.float32, device="cuda")
    ds.layer(sh, W, x, out, ws)
    xh = x.cpu().pin_memory()
    oh = torch.empty((1, cfg.D), dtype=torch.float32).pin_memory()
    ds.layer_hostio(sh, W, xh, oh, ws)
    ds.sync_status()
    assert torch.equal(oh, out.cpu())
    x2 = torch.cat([x, x])
    out2 = torch.empty((2, cfg.D), dtype=torch.float32, device="cuda")
    assert ds.layer_path(sh, 2) == ds.PATH_DECODE3
    ds.layer(sh, W, x2, out2, ws)
    ds.sync_status()
    assert torch.equal(out2[0], out2[1])
    ref = out2[0].cpu().numpy().astype(np.float64)
    check_close(out.cpu().numpy()[0], ref, DECODE_TOL, "stream vs three-kernel chain")


def test_q4k_mixed_stack_by_layer():
    """A mixed stack (Q2_K layers, then Q4_K layers, as in a "q2-q4" model)
    at full width, T=8, through ds_moe_stack_mixed: each layer against the
    oracle on the residual the GPU produced before it (as in the Q2_K stack
    test), then the four-layer call bit-identical to one call per layer."""
    from dataclasses import replace
    fmts = ["q2k", "q2k", "q4k", "q4k"]
    cfgs = [replace(dsgen.STACK, expert_fmt=f) for f in fmts]
    codes = [ds.DS_Q4_K if f == "q4k" else ds.DS_Q2_K for f in fmts]
    Ws = [synthetic.build_layer(c, l) for l, c in enumerate(cfgs)]
    sh = synthetic.shape_of(cfgs[0])
    ws = torch.empty(ds.workspace_bytes(sh, dsgen.STACK.T), dtype=torch.uint8, device="cuda")
    x0 = torch.from_numpy(dsgen.host_x(replace(dsgen.STACK, x_dtype="f32"))).cuda()
    x = x0.clone()
    checked = 0
    for l, c in enumerate(cfgs):
        x_in = x.cpu().numpy()
        ds.stack(sh, [Ws[l]], x, ws, formats=[codes[l]])
        ds.sync_status()
        got = x.cpu().numpy().astype(np.float64) - x_in
        lo = oracle.LayerOracle(c, l)
        r64 = oracle.as_f64(oracle.rmsnorm_bf16(x_in), "bf16")
        res, _, _, L = lo.forward(r64)
        keep = oracle.min_top_gap(L, c.k) >= oracle.GAP
        ref = (x_in.astype(np.float64) + res).astype(np.float32).astype(np.float64) - x_in
        check_close(got[keep], ref[keep], DECODE_TOL, f"mixed stack layer {l} {fmts[l]}")
        checked += int(keep.sum())
    assert checked >= len(cfgs) * dsgen.STACK.T - 2
    xa = x0.clone()
    ds.stack(sh, Ws, xa, ws, formats=codes)
    ds.sync_status()
    assert torch.equal(xa, x)
