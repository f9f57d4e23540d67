"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each check is chosen so that a plausible mistake in the oracle (a swapped
nibble, a wrong code bit order, a dropped min term, gate/up swapped, a wrong
tie rule, a non-stable permutation, a missing shared expert) fails at least
one of them.  None of these tests touches a GPU.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import dsgen
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def facts():
    with open(os.path.join(GOLD, "pages_facts.json")) as f:
        return json.load(f)


# ------------------------------------------------------------ printed sizes --

def test_block_size_matches_pages():
    f = facts()["q2k_block"]
    assert oracle.q2k_bytes(1, 256) == f["bytes_per_block"]
    assert f["bytes_per_block"] * 8 / f["weights_per_block"] == f["bits_per_weight"]
    # 16 scale/min bytes + 64 code bytes + fp16 d + fp16 dmin
    assert 16 + f["weights_per_block"] * 2 // 8 + f["scale_bytes"] + f["min_bytes"] == 84
    assert f["sub_blocks"] * f["weights_per_sub_block"] == f["weights_per_block"]
    # rows pad to whole blocks
    assert oracle.q2k_bytes(3, 257) == 3 * 2 * 84
    assert oracle.q2k_bytes(5, 128) == 5 * 84


def test_parameter_arithmetic_matches_pages():
    s = facts()["flash_shape"]
    p = facts()["param_counts"]
    per_expert = 3 * s["n_embd"] * s["n_ff_exp"]
    assert per_expert == 25_165_824
    assert round(per_expert / 1e6, 1) == p["per_expert_millions_rounded_1dp"]
    per_layer = per_expert * s["n_expert"]
    assert round(per_layer / 1e9, 2) == p["per_layer_billions_rounded_2dp"]
    assert round(per_layer * s["n_layer"] / 1e9) == p["model_billions_rounded_0dp"]
    # packed sizes of one expert / one layer / 43 layers at 84 bytes per 256 weights
    eb = oracle.lib().oracle_expert_bytes(s["n_embd"], s["n_ff_exp"])
    assert eb == 8_257_536 == per_expert // 256 * 84
    assert eb * s["n_expert"] == 2_113_929_216
    assert eb * s["n_expert"] * s["n_layer"] == 90_898_956_288
    assert dsgen.DECODE1.expert_bytes == eb
    # the same expert in 144-byte Q4_K blocks (4.5 bits per weight)
    eb4 = oracle.lib().oracle_expert_bytes_fmt(1, s["n_embd"], s["n_ff_exp"])
    assert eb4 == per_expert // 256 * 144 == 14_155_776
    assert oracle.lib().oracle_expert_bytes_fmt(0, s["n_embd"], s["n_ff_exp"]) == eb
    assert dsgen.DECODE1_Q4K.expert_bytes == eb4


# ------------------------------------------------------------------- fp16 --

@pytest.mark.parametrize("bits", [0x0000, 0x0001, 0x03FF, 0x0400, 0x3555, 0x3C00, 0x3C01, 0x7BFF,
                                  0x8001, 0xC000, 0xBC00])
def test_fp16_value_matches_numpy(bits):
    ref = float(np.array([bits], np.uint16).view(np.float16)[0])
    assert oracle.fp16_value(bits) == ref


def test_bf16_round_ties_to_even_and_neighbours():
    one = 1.0
    ulp = 2.0 ** -7
    assert oracle.bf16_round(one) == 0x3F80
    assert oracle.bf16_round(one + ulp / 2) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_round(one + 3 * ulp / 2) == 0x3F82      # tie -> even (1 + 2ulp)
    assert oracle.bf16_round(one + ulp / 2 + 1e-12) == 0x3F81  # above the tie
    assert oracle.bf16_round(-2.0) == 0xC000
    # agrees with a brute-force nearest search over all bf16 values near v
    rng = np.random.default_rng(5)
    for v in rng.normal(size=200) * 10.0 ** rng.integers(-30, 30, 200):
        b = oracle.bf16_round(float(v))
        cand = np.arange(max(b - 2, 0), b + 3, dtype=np.uint32)
        vals = (cand << 16).view(np.float32).astype(np.float64)
        assert abs(float(dsgen.bf16_bits_to_f32(np.array([b], np.uint16))[0]) - v) <= np.min(np.abs(vals - v))


# -------------------------------------------------------------- dequantise --

def handbuilt_block(d_bits, dmin_bits, sc, m, q):
    blk = np.zeros(84, np.uint8)
    for s in range(16):
        blk[s] = sc[s] | (m[s] << 4)
    for j in range(256):
        blk[16 + j // 4] |= q[j] << (2 * (j % 4))
    blk[80], blk[81] = d_bits & 0xFF, d_bits >> 8
    blk[82], blk[83] = dmin_bits & 0xFF, dmin_bits >> 8
    return blk


def test_dequant_closed_form_handbuilt():
    # d = 1 (0x3C00), dmin = 0.5 (0x3800), sc = 3, m = 2  ->  w = 3q - 1 = -1, 2, 5, 8
    sc = [3] * 16
    m = [2] * 16
    q = [j % 4 for j in range(256)]
    blk = handbuilt_block(0x3C00, 0x3800, sc, m, q)
    w = oracle.dequantize(blk, 1, 256)[0]
    assert list(w[:8]) == [-1.0, 2.0, 5.0, 8.0, -1.0, 2.0, 5.0, 8.0]
    # per-sub-block scale/min nibbles: sub-block 5 gets sc = 7 (low), m = 1 (high)
    sc[5], m[5] = 7, 1
    q2 = [3 if j == 16 * 5 + 2 else 0 for j in range(256)]
    blk = handbuilt_block(0x3C00, 0x3800, sc, m, q2)
    w = oracle.dequantize(blk, 1, 256)[0]
    assert w[16 * 5 + 2] == 1.0 * 7 * 3 - 0.5 * 1
    assert w[16 * 5 + 3] == -0.5
    assert w[0] == -1.0
    # code bit order: weight j lives at byte 16 + j//4, bits 2*(j%4)
    q3 = [0] * 256
    q3[6] = 2  # byte 17, bits 4-5
    blk = handbuilt_block(0x3C00, 0x0000, [1] * 16, [0] * 16, q3)
    assert blk[17] == 2 << 4
    w = oracle.dequantize(blk, 1, 256)[0]
    assert w[6] == 2.0 and np.count_nonzero(w) == 1


def test_dequant_matches_fraction_arithmetic_random_blocks():
    rng = np.random.default_rng(1)
    for _ in range(20):
        blk = rng.integers(0, 256, 84).astype(np.uint8)
        # keep d, dmin finite and non-negative
        for o in (80, 82):
            v = int(rng.integers(0, 0x7BFF))
            blk[o], blk[o + 1] = v & 0xFF, v >> 8
        w = oracle.dequantize(blk, 1, 256)[0]
        d = _h(int(blk[80]) | (int(blk[81]) << 8))
        dm = _h(int(blk[82]) | (int(blk[83]) << 8))
        for j in range(0, 256, 7):
            s = j // 16
            q = (int(blk[16 + j // 4]) >> (2 * (j % 4))) & 3
            exact = d * (int(blk[s]) & 15) * q - dm * (int(blk[s]) >> 4)
            assert Fraction(w[j]) == exact


# --------------------------------------------------------------- quantise --

def _fields(blk):
    sc = [int(b) & 15 for b in blk[:16]]
    m = [int(b) >> 4 for b in blk[:16]]
    q = [(int(blk[16 + j // 4]) >> (2 * (j % 4))) & 3 for j in range(256)]
    d_bits = int(blk[80]) | (int(blk[81]) << 8)
    dm_bits = int(blk[82]) | (int(blk[83]) << 8)
    return sc, m, q, d_bits, dm_bits


def _h(bits):
    return Fraction(float(np.array([bits], np.uint16).view(np.float16)[0]))


@pytest.mark.parametrize("scale", [0.02, 1.0, 37.0, 1e-4])
def test_quantizer_invariants_exact(scale):
    """Range coverage, minimality of every scale, and the half-step error bound,
    all checked in exact rational arithmetic."""
    rng = np.random.default_rng(int(scale * 1e4) + 3)
    x = (rng.normal(size=(6, 256)) * scale).astype(np.float32)
    x[1, :16] = np.abs(x[1, :16])       # a sub-block with no negative value
    x[2, 32:48] = -np.abs(x[2, 32:48])  # a sub-block with no positive value
    x[3, 64:80] = 0.0                   # an all-zero sub-block
    q = oracle.quantize(x)
    deq = oracle.dequantize(q, 6, 256)
    for r in range(6):
        sc, m, qq, d_bits, dm_bits = _fields(q[r])
        d, dmin = _h(d_bits), _h(dm_bits)
        X = [Fraction(float(v)) for v in x[r]]
        lo = [min(Fraction(0), min(X[16 * s:16 * s + 16])) for s in range(16)]
        hi = [max(X[16 * s:16 * s + 16]) for s in range(16)]
        assert 15 * dmin >= max(-l for l in lo)
        if dm_bits > 0:
            assert 15 * _h(dm_bits - 1) < max(-l for l in lo)  # smallest such fp16
        b = []
        for s in range(16):
            assert 0 <= m[s] <= 15 and 0 <= sc[s] <= 15
            assert m[s] * dmin >= -lo[s]
            if m[s] > 0:
                assert (m[s] - 1) * dmin < -lo[s]
            b.append(m[s] * dmin)
        assert all(45 * d >= hi[s] + b[s] for s in range(16))
        if d_bits > 0:
            assert any(45 * _h(d_bits - 1) < hi[s] + b[s] for s in range(16))
        for s in range(16):
            assert 3 * d * sc[s] >= hi[s] + b[s]
            if sc[s] > 0:
                assert 3 * d * (sc[s] - 1) < hi[s] + b[s]
            step = d * sc[s]
            for j in range(16 * s, 16 * s + 16):
                assert -b[s] <= X[j] <= -b[s] + 3 * step       # inside the 4-level range
                w = Fraction(deq[r, j])
                assert abs(X[j] - w) <= step / 2                  # nearest level
                if step > 0:  # round-half-up code choice, exactly
                    t = (X[j] + b[s]) / step
                    assert qq[j] == min(3, math.floor(t + Fraction(1, 2)))


def test_quantizer_all_zero_block():
    q = oracle.quantize(np.zeros((2, 256), np.float32))
    assert not q.any()


def test_quantizer_roundtrip_on_grid_is_byte_exact():
    """A block whose values already lie on its own grid (max scale and min 15,
    each sub-block using codes 0 and 3) quantises back to the same bytes."""
    rng = np.random.default_rng(7)
    for trial in range(25):
        d_bits = int(rng.integers(0x1000, 0x3000))
        dm_bits = int(rng.integers(0x1000, 0x3000))
        sc = list(rng.integers(1, 16, 16))
        m = list(rng.integers(0, 16, 16))
        sc[int(rng.integers(16))] = 15
        m[int(rng.integers(16))] = 15
        q = list(rng.integers(0, 4, 256))
        for s in range(16):
            q[16 * s], q[16 * s + 1] = 0, 3
        blk = handbuilt_block(d_bits, dm_bits, sc, m, q)
        w = oracle.dequantize(blk, 1, 256)
        w32 = w.astype(np.float32)
        assert np.array_equal(w32.astype(np.float64), w)  # grid values are fp32-exact here
        again = oracle.quantize(w32)
        assert np.array_equal(again[0], blk), trial


def test_quantizer_zero_pads_short_rows():
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(4, 128)) * 0.02).astype(np.float32)
    q = oracle.quantize(x)
    assert q.shape == (4, 84)
    for r in range(4):
        sc, m, _, _, _ = _fields(q[r])
        assert sc[8:] == [0] * 8 and m[8:] == [0] * 8  # padded sub-blocks
    padded = np.concatenate([x, np.zeros((4, 128), np.float32)], axis=1)
    assert np.array_equal(oracle.quantize(padded), q)
    assert oracle.dequantize(q, 4, 128).shape == (4, 128)


def test_quantizer_rejects_non_finite_and_out_of_domain():
    for bad in (np.nan, np.inf, -np.inf, 65505.0, -70000.0):
        x = np.zeros((1, 256), np.float32)
        x[0, 3] = bad
        with pytest.raises(ValueError):
            oracle.quantize(x)
    x = np.zeros((1, 256), np.float32)
    x[0, 3] = -65504.0  # the largest fp16 magnitude is inside the domain
    q = oracle.quantize(x)
    # dmin = fp16 >= 65504/15 = 4368, m = 15: the low level is -65520 (half-step bound holds)
    assert oracle.dequantize(q, 1, 256)[0, 3] == -65520.0


# ---------------------------------------------------------------- routing --

def _brute_topk(L, k):
    """Sort all experts by (-logit, index) with a library sort."""
    order = np.lexsort((np.arange(L.shape[1])[None, :].repeat(L.shape[0], 0), -L), axis=1)
    return order[:, :k]


def test_select_matches_brute_force_sort_with_ties():
    rng = np.random.default_rng(3)
    L = rng.normal(size=(64, 256))
    L[0, [3, 9, 200]] = 10.0          # an exact three-way tie at the top
    L[1, :] = 0.5                      # all equal: ids must be 0..k-1
    L[2, [7, 5]] = 4.0                 # tie straddling the cut is resolved by index
    ids, w = oracle.select(L, 6)
    lex = np.lexsort((np.tile(np.arange(256), (64, 1)), -L), axis=1)[:, :6]
    assert np.array_equal(ids, lex)
    assert list(ids[0, :3]) == [3, 9, 200]
    assert list(ids[1]) == [0, 1, 2, 3, 4, 5]
    assert list(ids[2, :2]) == [5, 7]
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=4e-16)
    # weights equal the full softmax renormalised over the selected experts
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    sel = np.take_along_axis(p, ids, 1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13, atol=0)
    # descending weight order follows descending logit order
    assert np.all(np.diff(w, axis=1) <= 0)


def test_select_k_equals_E_is_full_softmax_and_scale():
    rng = np.random.default_rng(4)
    L = rng.normal(size=(5, 16))
    ids, w = oracle.select(L, 16)
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(np.take_along_axis(p, ids, 1), w, rtol=1e-14, atol=0)
    _, w15 = oracle.select(L, 16, routed_scale=1.5)
    assert np.allclose(w15, 1.5 * w, rtol=1e-15, atol=0)


def test_select_logit_scale():
    """The logit scale ([UDS] 5.3.5's reading of the 1.5 as a scale applied
    before the softmax): the picks do not change; for k = 2 the first weight
    is the logistic function of s times the gap (closed form); s = 1 is the
    plain softmax; a large s puts all the weight on the top logit."""
    rng = np.random.default_rng(11)
    L = rng.normal(size=(6, 40))
    ids1, w1 = oracle.select(L, 6)
    for s_ in (0.5, 1.5, 3.0):
        ids_s, w_s = oracle.select(L, 6, logit_scale=s_)
        assert np.array_equal(ids_s, ids1)
        assert np.allclose(w_s.sum(1), 1.0, rtol=0, atol=1e-14)
    _, w_one = oracle.select(L, 6, logit_scale=1.0)
    assert np.array_equal(w_one, w1)
    ids2, w2 = oracle.select(L, 2, logit_scale=1.5)
    gap = np.take_along_axis(L, ids2[:, :1], 1) - np.take_along_axis(L, ids2[:, 1:], 1)
    assert np.allclose(w2[:, :1], 1.0 / (1.0 + np.exp(-1.5 * gap)), rtol=1e-14, atol=0)
    Ls = np.array([[0.0, 3.0, 1.0, 2.0]])
    _, w_big = oracle.select(Ls, 3, logit_scale=60.0)
    assert w_big[0, 0] >= 1 - 1e-15 and w_big[0, 1] < 1e-25 and w_big[0, 2] < 1e-50
    _, w_mix = oracle.select(L, 6, routed_scale=1.5, logit_scale=1.5)
    _, w_l = oracle.select(L, 6, logit_scale=1.5)
    assert np.allclose(w_mix, 1.5 * w_l, rtol=1e-15, atol=0)


def test_select_bias_for_selection_only():
    """A router bias that steers the selection only: the picks are those of
    the biased logits, and the weights are the softmax of the selected logits
    with the bias taken back out (k = 2: the logistic function of the
    unbiased gap); a zero bias changes nothing."""
    rng = np.random.default_rng(13)
    L0 = rng.normal(size=(7, 24))
    b = -1.1 * np.log(rng.permutation(24) + 1.0)
    Lb = L0 + b
    ids_b, w_b = oracle.select(Lb, 6)
    ids_s, w_s = oracle.select(Lb, 6, unbias=b)
    assert np.array_equal(ids_s, ids_b)
    assert np.allclose(w_s.sum(1), 1.0, rtol=0, atol=1e-14)
    assert not np.allclose(w_s, w_b)
    u = np.take_along_axis(L0, ids_s, 1)
    p = np.exp(u - u.max(1, keepdims=True))
    assert np.allclose(w_s, p / p.sum(1, keepdims=True), rtol=1e-13, atol=0)
    ids2, w2 = oracle.select(Lb, 2, unbias=b)
    gap = np.take_along_axis(L0, ids2[:, :1], 1) - np.take_along_axis(L0, ids2[:, 1:], 1)
    assert np.allclose(w2[:, :1], 1.0 / (1.0 + np.exp(-gap)), rtol=1e-13, atol=0)
    _, w_zero = oracle.select(Lb, 6, unbias=np.zeros(24))
    assert np.array_equal(w_zero, w_b)


def test_route_matches_stable_sort():
    rng = np.random.default_rng(5)
    for T, k, E in ((1, 6, 256), (37, 6, 256), (8, 2, 16), (200, 4, 7)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm, pos = oracle.route(ids, E)
        assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm, np.argsort(ids.ravel(), kind="stable"))
        assert np.array_equal(perm[pos], np.arange(T * k))


def test_router_logits_brute_force():
    rng = np.random.default_rng(6)
    x = rng.normal(size=(3, 40))
    wr = rng.normal(size=(5, 40))
    b = rng.normal(size=5)
    L = oracle.router_logits(x, wr, b)
    for t in range(3):
        for e in range(5):
            assert math.isclose(L[t, e], math.fsum(x[t] * wr[e]) + b[e], rel_tol=1e-13, abs_tol=1e-13)


# ------------------------------------------------------------------ layer --

def _silu(z):
    return z / (1.0 + np.exp(-z))


def _rand_experts(rng, E, D, F, sigma=0.02):
    blobs, deq = {}, {}
    for e in range(E):
        g = (rng.normal(size=(F, D)) * sigma).astype(np.float32)
        u = (rng.normal(size=(F, D)) * sigma).astype(np.float32)
        dn = (rng.normal(size=(D, F)) * sigma).astype(np.float32)
        qg, qu, qd = oracle.quantize(g), oracle.quantize(u), oracle.quantize(dn)
        blobs[e] = np.concatenate([qg.ravel(), qu.ravel(), qd.ravel()])
        deq[e] = (oracle.dequantize(qg, F, D), oracle.dequantize(qu, F, D), oracle.dequantize(qd, D, F))
    return blobs, deq


def test_swiglu_closed_form_handbuilt_expert():
    """One expert with gate row 0 = e_0, up row 0 = 2 e_0 and down column 0 = 1:
    y_d = SiLU(x_0) * 2 x_0 for every d (gate and up are not interchangeable)."""
    D, F = 256, 256
    one = handbuilt_block(0x3C00, 0, [1] * 16, [0] * 16, [1] + [0] * 255)   # w_0 = 1
    two = handbuilt_block(0x4000, 0, [1] * 16, [0] * 16, [1] + [0] * 255)   # w_0 = 2
    zero = np.zeros(84, np.uint8)
    gate = np.stack([one] + [zero] * (F - 1))
    up = np.stack([two] + [zero] * (F - 1))
    down = np.stack([one] * D)
    blob = np.concatenate([gate.ravel(), up.ravel(), down.ravel()])
    x = np.zeros((3, D))
    x[:, 0] = [2.0, -1.5, 0.0]
    ids = np.zeros((3, 1), np.int32)
    out = oracle.moe_layer(x, {0: blob}, None, ids, np.ones((3, 1)), D, 1, F, 0)
    for t, x0 in enumerate([2.0, -1.5, 0.0]):
        expect = x0 / (1 + math.exp(-x0)) * 2 * x0
        assert np.allclose(out[t], expect, rtol=1e-15, atol=0)
    assert out[0, 0] != pytest.approx((2 * 2 / (1 + math.exp(-4))) * 2)  # swapped gate/up differs


def test_layer_top1_single_expert_is_swiglu_ffn():
    rng = np.random.default_rng(8)
    D, F = 256, 128
    blobs, deq = _rand_experts(rng, 1, D, F)
    x = rng.normal(size=(4, D))
    ids = np.zeros((4, 1), np.int32)
    out = oracle.moe_layer(x, blobs, None, ids, np.ones((4, 1)), D, 1, F, 0)
    g, u, dn = deq[0]
    ref = (_silu(x @ g.T) * (x @ u.T)) @ dn.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)


def test_layer_k_equals_E_is_dense_weighted_sum():
    rng = np.random.default_rng(9)
    D, F, E, T = 256, 128, 5, 6
    blobs, deq = _rand_experts(rng, E, D, F)
    x = rng.normal(size=(T, D))
    wr = rng.normal(size=(E, D)) * 0.05
    L = oracle.router_logits(x, wr)
    ids, w = oracle.select(L, E)
    out = oracle.moe_layer(x, blobs, None, ids, w, D, E, F, 0)
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = np.zeros((T, D))
    for e in range(E):
        g, u, dn = deq[e]
        ref += p[:, e:e + 1] * ((_silu(x @ g.T) * (x @ u.T)) @ dn.T)
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-14)


def test_layer_k1_is_argmax_expert_and_shared_is_added_unweighted():
    rng = np.random.default_rng(10)
    D, F, E, T, Fs = 256, 128, 4, 5, 64
    blobs, deq = _rand_experts(rng, E, D, F)
    x = rng.normal(size=(T, D))
    wr = rng.normal(size=(E, D)) * 0.05
    sg, su = rng.normal(size=(Fs, D)) * 0.02, rng.normal(size=(Fs, D)) * 0.02
    sd = rng.normal(size=(D, Fs)) * 0.02
    L = oracle.router_logits(x, wr)
    ids, w = oracle.select(L, 1)
    assert np.array_equal(ids[:, 0], np.argmax(L, 1))
    assert np.all(w == 1.0)
    out = oracle.moe_layer(x, blobs, (sg, su, sd), ids, w, D, E, F, Fs)
    shared = (_silu(x @ sg.T) * (x @ su.T)) @ sd.T
    for t in range(T):
        g, u, dn = deq[int(ids[t, 0])]
        ref = (_silu(x[t] @ g.T) * (x[t] @ u.T)) @ dn.T + shared[t]
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-14)


def test_layer_token_permutation_invariance_bit_exact():
    rng = np.random.default_rng(11)
    D, F, E, T, k = 256, 128, 8, 9, 3
    blobs, _ = _rand_experts(rng, E, D, F)
    x = rng.normal(size=(T, D))
    wr = rng.normal(size=(E, D)) * 0.05
    ids, w = oracle.select(oracle.router_logits(x, wr), k)
    out = oracle.moe_layer(x, blobs, None, ids, w, D, E, F, 0)
    pi = rng.permutation(T)
    ids2, w2 = oracle.select(oracle.router_logits(x[pi], wr), k)
    out2 = oracle.moe_layer(x[pi], blobs, None, ids2, w2, D, E, F, 0)
    assert np.array_equal(out2, out[pi])


def test_layer_missing_selected_expert_is_an_error():
    D, F = 256, 128
    x = np.zeros((1, D))
    with pytest.raises(ValueError):
        oracle.moe_layer(x, {}, None, np.zeros((1, 1), np.int32), np.ones((1, 1)), D, 1, F, 0)


# ------------------------------------------------------------------ stack --

def test_rmsnorm_constant_vector_is_unit():
    x = np.full((2, 4096), 3.0, np.float32)
    x[1] = -0.25
    r = oracle.rmsnorm_bf16(x)
    assert np.all(r[0] == 0x3F80) and np.all(r[1] == 0xBF80)


def test_rmsnorm_matches_definition():
    rng = np.random.default_rng(12)
    x = rng.normal(size=(3, 512)).astype(np.float32) * 3
    r = dsgen.bf16_bits_to_f32(oracle.rmsnorm_bf16(x)).astype(np.float64)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt((x64 ** 2).mean(1, keepdims=True) + 1e-6)
    assert np.all(np.abs(r - ref) <= np.abs(ref) * 2.0 ** -8)


def test_zero_experts_leave_residual_unchanged():
    D, F, E = 256, 128, 4
    z = np.zeros(oracle.lib().oracle_expert_bytes(D, F), np.uint8)
    x = np.random.default_rng(13).normal(size=(2, D)).astype(np.float32)
    r = dsgen.bf16_bits_to_f32(oracle.rmsnorm_bf16(x)).astype(np.float64)
    ids, w = oracle.select(np.zeros((2, E)), 2)
    out = oracle.moe_layer(r, {e: z for e in range(E)}, None, ids, w, D, E, F, 0)
    assert not out.any()
    assert np.array_equal((x.astype(np.float64) + out).astype(np.float32), x)


# -------------------------------------------------------- workload recipe --

def test_tiny_config_resampling_leaves_clear_gaps():
    cfg = dsgen.TINY
    lo = oracle.LayerOracle(cfg)
    att = oracle.resample_attempts(cfg, lo)
    x = oracle.as_f64(dsgen.host_x(cfg, att), cfg.x_dtype)
    assert np.all(oracle.min_top_gap(lo.logits(x), cfg.k) >= oracle.GAP)
    out, ids, w, _ = lo.forward(x)
    assert out.shape == (cfg.T, cfg.D) and np.isfinite(out).all()
    assert np.all(np.diff(ids, axis=1) != 0)


# ------------------------------------------------------------------- Q4_K --
# The 144-byte Q4_K block of "Understanding Dwarf Star" 2.3.2 (the next
# expert format); readings of the packing as stated in the oracle.

def q4k_handbuilt(d_bits, dm_bits, sc, m, q):
    """A Q4_K block from its fields, packed here independently of the oracle:
    fp16 d, fp16 dmin, the sixteen 6-bit fields (sc_0..7, m_0..7) as a 96-bit
    little-endian integer, codes two per byte with the even value low."""
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, d_bits >> 8
    blk[2], blk[3] = dm_bits & 0xFF, dm_bits >> 8
    bits = 0
    for i, v in enumerate(list(sc) + list(m)):
        assert 0 <= v < 64
        bits |= int(v) << (6 * i)
    blk[4:16] = np.frombuffer(bits.to_bytes(12, "little"), np.uint8)
    for j in range(256):
        blk[16 + j // 2] |= int(q[j]) << (4 * (j % 2))
    return blk


def q4k_fields(blk):
    bits = int.from_bytes(bytes(blk[4:16]), "little")
    f = [(bits >> (6 * i)) & 63 for i in range(16)]
    q = [(int(blk[16 + j // 2]) >> (4 * (j % 2))) & 15 for j in range(256)]
    return f[:8], f[8:], q, int(blk[0]) | (int(blk[1]) << 8), int(blk[2]) | (int(blk[3]) << 8)


def test_q4k_block_size_matches_pages():
    f = facts()["q4k_block"]
    assert oracle.q4k_bytes(1, 256) == f["bytes_per_block"] == 144
    assert f["bytes_per_block"] * 8 / f["weights_per_block"] == f["bits_per_weight"] == 4.5
    assert f["sub_blocks"] * f["weights_per_sub_block"] == 256
    assert f["scales_offset"] + f["scales_bytes"] == f["codes_offset"]
    assert f["codes_offset"] + f["codes_bytes"] == f["bytes_per_block"]
    assert f["scales_bytes"] * 8 == 2 * f["sub_blocks"] * 6      # 8 scales + 8 mins, 6 bits each
    assert f["codes_bytes"] * 8 == 4 * f["weights_per_block"]     # 4-bit values
    assert oracle.q4k_bytes(3, 257) == 3 * 2 * 144


def test_q4k_dequant_closed_form_handbuilt():
    # d = 1, dmin = 0.5, sc = 3, m = 2  ->  w = 3q - 1 for q = 0..15
    q = [j % 16 for j in range(256)]
    blk = q4k_handbuilt(0x3C00, 0x3800, [3] * 8, [2] * 8, q)
    w = oracle.dequantize_q4k(blk, 1, 256)[0]
    assert list(w[:16]) == [3.0 * v - 1.0 for v in range(16)]
    # 6-bit fields beyond a nibble, per sub-block: sub-block 5 has sc = 40, m = 33
    sc, m = [3] * 8, [2] * 8
    sc[5], m[5] = 40, 33
    blk = q4k_handbuilt(0x3C00, 0x3800, sc, m, q)
    w = oracle.dequantize_q4k(blk, 1, 256)[0]
    assert w[32 * 5 + 7] == 40.0 * 7 - 0.5 * 33
    assert w[32 * 4 + 7] == 3.0 * 7 - 1.0
    # the packing itself: field 0 in the low bits of byte 4, field 8 (m_0) at bit 48
    blk = q4k_handbuilt(0x3C00, 0x3C00, [63, 0, 0, 0, 0, 0, 0, 0], [1, 0, 0, 0, 0, 0, 0, 0], [0] * 256)
    assert blk[4] == 0x3F and blk[5] == 0 and blk[10] == 1 and not blk[11:16].any()
    # code order: value 1 is the high nibble of byte 16
    q1 = [0] * 256
    q1[1] = 7
    blk = q4k_handbuilt(0x3C00, 0x0000, [1] * 8, [0] * 8, q1)
    assert blk[16] == 0x70
    w = oracle.dequantize_q4k(blk, 1, 256)[0]
    assert w[1] == 7.0 and np.count_nonzero(w) == 1


def test_q4k_dequant_matches_fraction_arithmetic_random_blocks():
    rng = np.random.default_rng(21)
    for _ in range(20):
        blk = rng.integers(0, 256, 144).astype(np.uint8)
        for o in (0, 2):
            v = int(rng.integers(0, 0x7BFF))
            blk[o], blk[o + 1] = v & 0xFF, v >> 8
        w = oracle.dequantize_q4k(blk, 1, 256)[0]
        sc, m, q, d_bits, dm_bits = q4k_fields(blk)
        d, dm = _h(d_bits), _h(dm_bits)
        for j in range(0, 256, 5):
            s = j // 32
            assert Fraction(w[j]) == d * sc[s] * q[j] - dm * m[s]


@pytest.mark.parametrize("scale", [0.02, 1.0, 300.0, 1e-4])
def test_q4k_quantizer_invariants_exact(scale):
    """Minimality of every scale, range coverage, the half-step bound and the
    round-half-up code, in exact rational arithmetic."""
    rng = np.random.default_rng(int(scale * 1e4) + 5)
    x = (rng.normal(size=(5, 256)) * scale).astype(np.float32)
    x[1, :32] = np.abs(x[1, :32])
    x[2, 64:96] = -np.abs(x[2, 64:96])
    x[3, 128:160] = 0.0
    qb = oracle.quantize_q4k(x)
    deq = oracle.dequantize_q4k(qb, 5, 256)
    for r in range(5):
        sc, m, qq, d_bits, dm_bits = q4k_fields(qb[r])
        d, dmin = _h(d_bits), _h(dm_bits)
        X = [Fraction(float(v)) for v in x[r]]
        lo = [min(Fraction(0), min(X[32 * s:32 * s + 32])) for s in range(8)]
        hi = [max(X[32 * s:32 * s + 32]) for s in range(8)]
        assert 63 * dmin >= max(-l for l in lo)
        if dm_bits > 0:
            assert 63 * _h(dm_bits - 1) < max(-l for l in lo)
        b = []
        for s in range(8):
            assert m[s] * dmin >= -lo[s]
            if m[s] > 0:
                assert (m[s] - 1) * dmin < -lo[s]
            b.append(m[s] * dmin)
        assert all(945 * d >= hi[s] + b[s] for s in range(8))
        if d_bits > 0:
            assert any(945 * _h(d_bits - 1) < hi[s] + b[s] for s in range(8))
        for s in range(8):
            assert 15 * d * sc[s] >= hi[s] + b[s]
            if sc[s] > 0:
                assert 15 * d * (sc[s] - 1) < hi[s] + b[s]
            step = d * sc[s]
            for j in range(32 * s, 32 * s + 32):
                assert -b[s] <= X[j] <= -b[s] + 15 * step
                assert abs(X[j] - Fraction(deq[r, j])) <= step / 2
                if step > 0:
                    assert qq[j] == min(15, math.floor((X[j] + b[s]) / step + Fraction(1, 2)))


def test_q4k_quantizer_edge_cases():
    assert not oracle.quantize_q4k(np.zeros((2, 256), np.float32)).any()
    for bad in (np.nan, np.inf, 65505.0):
        x = np.zeros((1, 256), np.float32)
        x[0, 9] = bad
        with pytest.raises(ValueError):
            oracle.quantize_q4k(x)
    rng = np.random.default_rng(3)
    x = (rng.normal(size=(3, 128)) * 0.02).astype(np.float32)
    q = oracle.quantize_q4k(x)
    assert q.shape == (3, 144)
    for r in range(3):
        sc, m, _, _, _ = q4k_fields(q[r])
        assert sc[4:] == [0] * 4 and m[4:] == [0] * 4  # padded sub-blocks
    assert np.array_equal(oracle.quantize_q4k(np.concatenate([x, np.zeros((3, 128), np.float32)], 1)), q)


def test_q4k_quantizer_roundtrip_on_grid_is_byte_exact():
    """A block whose values lie on its own grid (a sub-block with scale 63,
    one with min 63, codes 0 and 15 in every sub-block) quantises back to the
    same bytes."""
    rng = np.random.default_rng(17)
    for trial in range(25):
        d_bits = int(rng.integers(0x2C00, 0x3000))   # d and dmin share an exponent:
        dm_bits = int(rng.integers(0x2C00, 0x3000))  # the grid values are fp32-exact
        sc = list(rng.integers(1, 64, 8))
        m = list(rng.integers(0, 64, 8))
        sc[int(rng.integers(8))] = 63
        m[int(rng.integers(8))] = 63
        q = list(rng.integers(0, 16, 256))
        for s in range(8):
            q[32 * s], q[32 * s + 1] = 0, 15
        blk = q4k_handbuilt(d_bits, dm_bits, sc, m, q)
        w = oracle.dequantize_q4k(blk, 1, 256)
        w32 = w.astype(np.float32)
        assert np.array_equal(w32.astype(np.float64), w)
        assert np.array_equal(oracle.quantize_q4k(w32)[0], blk), trial


def test_q4k_swiglu_closed_form_handbuilt_expert():
    """The hand-built SwiGLU expert again, stored as Q4_K blocks packed by
    the test: y_d = SiLU(x_0) * 2 x_0 for every d."""
    D, F = 256, 256
    e0 = [1] + [0] * 255
    one = q4k_handbuilt(0x3C00, 0, [1] * 8, [0] * 8, e0)   # w_0 = 1
    two = q4k_handbuilt(0x4000, 0, [1] * 8, [0] * 8, e0)   # w_0 = 2
    zero = np.zeros(144, np.uint8)
    gate = np.stack([one] + [zero] * (F - 1))
    up = np.stack([two] + [zero] * (F - 1))
    down = np.stack([one] * D)
    blob = np.concatenate([gate.ravel(), up.ravel(), down.ravel()])
    assert blob.size == oracle.lib().oracle_expert_bytes_fmt(1, D, F)
    x = np.zeros((3, D))
    x[:, 0] = [2.0, -1.5, 0.0]
    out = oracle.moe_layer(x, {0: blob}, None, np.zeros((3, 1), np.int32), np.ones((3, 1)), D, 1,
                           F, 0, fmt="q4k")
    for t, x0 in enumerate([2.0, -1.5, 0.0]):
        assert np.allclose(out[t], x0 / (1 + math.exp(-x0)) * 2 * x0, rtol=1e-15, atol=0)


def test_q4k_layer_top1_single_expert_is_swiglu_ffn():
    rng = np.random.default_rng(12)
    D, F = 256, 128
    g, u = (rng.normal(size=(F, D)) * 0.02).astype(np.float32), (rng.normal(size=(F, D)) * 0.02).astype(np.float32)
    dn = (rng.normal(size=(D, F)) * 0.02).astype(np.float32)
    qg, qu, qd = oracle.quantize_q4k(g), oracle.quantize_q4k(u), oracle.quantize_q4k(dn)
    blob = np.concatenate([qg.ravel(), qu.ravel(), qd.ravel()])
    G, U, DN = (oracle.dequantize_q4k(qg, F, D), oracle.dequantize_q4k(qu, F, D),
                oracle.dequantize_q4k(qd, D, F))
    x = rng.normal(size=(4, D))
    out = oracle.moe_layer(x, {0: blob}, None, np.zeros((4, 1), np.int32), np.ones((4, 1)), D, 1,
                           F, 0, fmt="q4k")
    ref = (_silu(x @ G.T) * (x @ U.T)) @ DN.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)
    # 4-bit codes track the fp32 weights closer than 2-bit ones
    e4 = np.abs(G - g).max() / np.abs(g).max()
    e2 = np.abs(oracle.dequantize(oracle.quantize(g), F, D) - g).max() / np.abs(g).max()
    assert e4 < e2 / 3
