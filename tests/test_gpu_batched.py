"""Parity of the batched decode path (4..16 tokens), of every selection
implementation on exact ties and of every path with more than 256 experts,
through the C ABI, against the fp64 oracle.

Batched decode (4..16 tokens): routed experts as exact integer dots on 16-bit fixed-point
activations, the shared expert on the tensor cores with exact bf16 products;
outputs within the decode tolerance 2e-3 * rms(out_oracle), ids, counts,
offsets and the permutation bit-exact.

Exact ties: a router with one expert row duplicated gives two bit-equal
logits on both sides.  For one token the pair straddles the k-th place, so
the lower index must be selected and the higher left out ("Understanding
Dwarf Star", 5.3.2: the top-k experts; the tie rule is this library's
reading: ties go to the lower index).  Every other gap among a token's top
k + 1 logits is kept at 1e-4 or more, so ids and their order have one answer.
Each selection implementation meets it: the one-token kernel's router warp
(T = 1), the three-kernel chain's router warp (T = 3), the batched decode
kernel (T = 16), the small-batch route kernel (T = 33, fp32 inputs) and the
large-batch selection kernel behind the tensor-core router (T = 300).
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


def run(cfg, W, x, bias_select_only=0):
    T = x.shape[0]
    sh = synthetic.shape_of(cfg)
    sh.bias_select_only = bias_select_only
    ws = torch.empty(ds.workspace_bytes(sh, T), dtype=torch.uint8, device="cuda")
    out = torch.full((T, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    dbg = {"logits": torch.empty((T, cfg.E), dtype=torch.float32, device="cuda"),
           "ids": torch.empty((T, cfg.k), dtype=torch.int32, device="cuda"),
           "w": torch.empty((T, cfg.k), dtype=torch.float32, device="cuda"),
           "counts": torch.empty(cfg.E, dtype=torch.int32, device="cuda"),
           "offsets": torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda"),
           "perm": torch.empty(T * cfg.k, dtype=torch.int32, device="cuda")}
    ds.layer(sh, W, x, out, ws, debug=dbg)
    ds.sync_status()
    return out.cpu().numpy(), {k: v.cpu().numpy() for k, v in dbg.items()}


def close(got, ref, tol, what="out"):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.max(np.abs(got.astype(np.float64) - ref))
    print(f"{what}: max|err|/rms = {err / rms:.3e}")
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e}"


def parity(cfg, bias_select_only=0, W=None, path=ds.PATH_BATCHED_DECODE, tol=DECODE_TOL):
    lo = oracle.LayerOracle(cfg)
    att = oracle.resample_attempts(cfg, lo)
    x64 = oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype)
    W = synthetic.build_layer(cfg) if W is None else W
    assert ds.layer_path(synthetic.shape_of(cfg), cfg.T) == path
    out, dbg = run(cfg, W, synthetic.build_x(cfg, att), bias_select_only)
    L = lo.logits(x64)
    ids, w = oracle.select(L, cfg.k, 1.0, 1.0, lo.bias if bias_select_only else None)
    assert np.array_equal(dbg["ids"], ids)
    counts, offsets, perm, _ = oracle.route(ids, cfg.E)
    assert np.array_equal(dbg["counts"], counts)
    assert np.array_equal(dbg["offsets"], offsets)
    assert np.array_equal(dbg["perm"], perm)
    assert np.max(np.abs(dbg["w"] - w)) <= 1e-5
    res = oracle.moe_layer(x64, lo.experts(ids), lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs,
                           fmt=cfg.expert_fmt)
    close(out, res, tol, cfg.name)
    return out


def _w1024(T, Fs, k, E, zipf=0.0, seed=11):
    return replace(dsgen.TINY, name=f"batched D=1024 F=1024 T={T} Fs={Fs} k={k} E={E} zipf={zipf}",
                   T=T, D=1024, F=1024, E=E, k=k, Fs=Fs, shared_sigma=0.02, x_dtype="bf16",
                   router_dtype="bf16", router_sigma=0.02, zipf_s=zipf, seed=seed)


@pytest.mark.parametrize("T,Fs,k,E,zipf", [(4, 1024, 2, 16, 0.0), (5, 1024, 2, 16, 0.0), (13, 0, 6, 40, 0.0),
                                            (16, 1024, 4, 8, 0.0), (16, 2048, 6, 64, 1.1),
                                            (15, 1024, 16, 16, 0.0), (9, 1024, 1, 3, 0.0)])
def test_batched_decode_width_1024(T, Fs, k, E, zipf):
    """At width 1024: the smallest batches of the path (4, 5), no shared expert, every
    expert with many tokens (E = 8, k = 4, 16 tokens), a Zipf-skewed route,
    k = E, one expert per token with an odd expert count."""
    parity(_w1024(T, Fs, k, E, zipf))


@pytest.fixture(scope="module")
def flash_layer():
    cfg = replace(dsgen.DECODE1, T=8)
    return cfg, synthetic.build_layer(cfg)


@pytest.mark.parametrize("T", [4, 5, 8, 12, 16])
def test_batched_decode_flash(flash_layer, T):
    """The Flash layer at the batch sizes of the path: one K slice of n_embd
    per block up to 8 tokens, then two (partial sums in a fixed order)."""
    cfg, W = flash_layer
    parity(replace(cfg, T=T), W=W)


def test_batched_decode_zipf_select_only():
    cfg = replace(dsgen.DECODE32_ZIPF, T=16)
    parity(cfg, bias_select_only=1)


def test_batched_decode_batch_invariance(flash_layer):
    """Tokens of an 8-token batch equal the same tokens in a 5-token batch bit
    for bit (both one K slice); a 16-token batch (two slices) agrees with
    them at the decode tolerance."""
    cfg, W = flash_layer
    c16 = replace(cfg, T=16)
    xb = synthetic.build_x(c16)
    out8, _ = run(replace(cfg, T=8), W, xb[:8].contiguous())
    out5, _ = run(replace(cfg, T=5), W, xb[3:8].contiguous())
    assert np.array_equal(out5, out8[3:8])
    out16, _ = run(c16, W, xb)
    close(out8.astype(np.float64), out16[:8].astype(np.float64), DECODE_TOL, "8 vs 16 tokens")


# ------------------------------------------------------------ exact ties --

def _top_gaps_ok(L, k):
    """Per token: among the top k + 1 logits every gap is 0 (an exact
    duplicate) or at least the oracle's resampling gap."""
    s = -np.sort(-L, axis=1)[:, : k + 1]
    d = s[:, :-1] - s[:, 1:]
    return np.all((d == 0) | (d >= oracle.GAP), axis=1)


def tie_case(cfg):
    """(router override, attempts, token with the straddling tie, a, b): row b
    of the router set to row a, with a at place k-1 and b (a higher index)
    outside the top k for that token; other tokens resampled until their top
    k + 1 logits have no near-tie."""
    lo = oracle.LayerOracle(cfg)
    att = oracle.resample_attempts(cfg, lo)
    L0 = lo.logits(oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype))
    for t0 in range(cfg.T):
        order = np.lexsort((np.arange(cfg.E), -L0[t0]))
        a = int(order[cfg.k - 1])
        cand = [e for e in range(a + 1, cfg.E) if e not in set(order[: cfg.k + 1].tolist())]
        if cand:
            b = cand[0]
            break
    else:
        raise RuntimeError("no token admits a straddling tie")
    wr = dsgen.host_router(cfg).copy()
    wr[b] = wr[a]
    lo.wr = oracle.as_f64(wr, cfg.router_dtype)
    for _ in range(64):
        L = lo.logits(oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype))
        bad = ~_top_gaps_ok(L, cfg.k)
        bad[t0] = False
        if not bad.any():
            break
        att[bad] += 1
    else:
        raise RuntimeError("tie resampling did not converge")
    assert L[t0, a] == L[t0, b]
    return lo, wr, att, t0, a, b


def _tie_cfg(T, dtype="bf16", Fs=1024, k=4, E=16):
    return replace(dsgen.TINY, name=f"tie T={T} {dtype} Fs={Fs} k={k} E={E}", T=T, D=1024, F=1024, E=E,
                   k=k, Fs=Fs, shared_sigma=0.02, x_dtype=dtype, router_dtype=dtype, router_sigma=0.02,
                   seed=23)


@pytest.mark.parametrize("T,dtype,Fs,path", [(1, "bf16", 512, ds.PATH_STREAM), (3, "bf16", 512, ds.PATH_DECODE3),
                                             (16, "bf16", 1024, ds.PATH_BATCHED_DECODE),
                                             (33, "f32", 1024, ds.PATH_GROUPED_GEMV),
                                             (300, "bf16", 1024, ds.PATH_TENSOR_CORE)])
def test_exact_tie_goes_to_lower_index(T, dtype, Fs, path):
    cfg = _tie_cfg(T, dtype, Fs)
    lo, wr, att, t0, a, b = tie_case(cfg)
    W = synthetic.build_layer(cfg)
    W.router_w.copy_(torch.from_numpy(wr.view(np.int16) if dtype == "bf16" else wr).cuda())
    assert ds.layer_path(synthetic.shape_of(cfg), T) == path
    out, dbg = run(cfg, W, synthetic.build_x(cfg, att))
    assert dbg["logits"][t0, a] == dbg["logits"][t0, b], "duplicated router rows gave different logits"
    x64 = oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype)
    L = lo.logits(x64)
    ids, w = oracle.select(L, cfg.k)
    assert a in ids[t0] and b not in ids[t0]
    assert np.array_equal(dbg["ids"], ids)
    assert np.max(np.abs(dbg["w"] - w)) <= 1e-5
    both = [t for t in range(T) if a in ids[t] and b in ids[t]]
    for t in both:  # the pair inside the top k: the lower index first
        assert list(ids[t]).index(a) < list(ids[t]).index(b)
    print(f"T={T}: tie straddles place {cfg.k} for token {t0}; both selected for {len(both)} tokens")
    res = oracle.moe_layer(x64, lo.experts(ids), lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs)
    tol = DECODE_TOL if path != ds.PATH_TENSOR_CORE else 5e-3
    close(out, res, tol, f"tie T={T}")


# ------------------------------------------------------- many experts --

@pytest.mark.parametrize("E", [300, 1024])
@pytest.mark.parametrize("T,dtype,Fs,path", [(1, "bf16", 512, ds.PATH_STREAM), (3, "bf16", 512, ds.PATH_DECODE3),
                                             (8, "bf16", 1024, ds.PATH_BATCHED_DECODE),
                                             (33, "f32", 1024, ds.PATH_GROUPED_GEMV),
                                             (300, "bf16", 1024, ds.PATH_TENSOR_CORE)])
def test_more_than_256_experts(E, T, dtype, Fs, path):
    """Expert counts above 256 (the library takes up to 1024): every lane of a
    selecting warp holds more than eight logits, so each selection
    implementation takes its general scan instead of the sorted eight-per-lane
    lists; 300 is not a multiple of 32 (ragged last lanes)."""
    cfg = replace(_tie_cfg(T, dtype, Fs, 6, E), name=f"E={E} T={T} {dtype}", seed=29)
    parity(cfg, path=path, tol=DECODE_TOL if path != ds.PATH_TENSOR_CORE else 5e-3)
