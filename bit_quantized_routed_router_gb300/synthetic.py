"""Synthetic layers in device memory, for benchmarks and tests.

Weights come from the seeded generator (``gen/dsgen.py``, device fills) and
are packed by the library's own ``ds_moe_quantize_q2k`` (or ``_q4k``); nothing here
computes any part of the layer.
"""
from __future__ import annotations

import os
import sys

import torch

from . import DS_BF16, DS_F32, DS_Q2_K, DS_Q4_K, MoEShape, MoEWeights, quantize_q2k, quantize_q4k

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if os.path.join(_ROOT, "gen") not in sys.path:
    sys.path.insert(0, os.path.join(_ROOT, "gen"))
import dsgen  # noqa: E402


def shape_of(cfg) -> MoEShape:
    return MoEShape(cfg.D, cfg.E, cfg.F, cfg.Fs, cfg.k,
                    DS_BF16 if cfg.x_dtype == "bf16" else DS_F32,
                    DS_BF16 if cfg.router_dtype == "bf16" else DS_F32, 1.0,
                    expert_format=DS_Q4_K if cfg.expert_fmt == "q4k" else DS_Q2_K)


def build_layer(cfg, layer: int = 0, device="cuda") -> MoEWeights:
    """All weights of one synthetic layer resident on the device."""
    dev = torch.device(device)
    E, D, F, Fs = cfg.E, cfg.D, cfg.F, cfg.Fs
    if cfg.router_dtype == "bf16":
        wr = torch.empty((E, D), dtype=torch.int16, device=dev)
        dsgen.dev_fill(None, wr, E * D, cfg.seed, layer, dsgen.T_ROUTER_W, 0, cfg.router_sigma,
                       cfg.router_dist)
    else:
        wr = torch.empty((E, D), dtype=torch.float32, device=dev)
        dsgen.dev_fill(wr, None, E * D, cfg.seed, layer, dsgen.T_ROUTER_W, 0, cfg.router_sigma,
                       cfg.router_dist)
    b = dsgen.host_bias(cfg, layer)
    bias = None if b is None else torch.from_numpy(b).to(dev)
    sh = [None, None, None]
    if Fs:
        for i, (t, n) in enumerate(((dsgen.T_SHARED_GATE, (Fs, D)), (dsgen.T_SHARED_UP, (Fs, D)),
                                    (dsgen.T_SHARED_DOWN, (D, Fs)))):
            sh[i] = torch.empty(n, dtype=torch.int16, device=dev)
            dsgen.dev_fill(None, sh[i], n[0] * n[1], cfg.seed, layer, t, 0, cfg.shared_sigma)
    eb = cfg.expert_bytes
    experts = torch.empty(E * eb, dtype=torch.uint8, device=dev)
    gb = F * cfg.rows_blocks(D) * cfg.block_bytes
    quantize = quantize_q4k if cfg.expert_fmt == "q4k" else quantize_q2k
    tmp = torch.empty(max(F * D, D * F), dtype=torch.float32, device=dev)
    for e in range(E):
        for t, rows, cols, off in ((dsgen.T_EXPERT_GATE, F, D, 0), (dsgen.T_EXPERT_UP, F, D, gb),
                                   (dsgen.T_EXPERT_DOWN, D, F, 2 * gb)):
            m = tmp[: rows * cols]
            dsgen.dev_fill(m, None, rows * cols, cfg.seed, layer, t, e, cfg.expert_sigma)
            nbytes = rows * cfg.rows_blocks(cols) * cfg.block_bytes
            quantize(m.view(rows, cols), experts[e * eb + off: e * eb + off + nbytes])
    return MoEWeights(router_w=wr, experts=experts, router_bias=bias, shared_gate=sh[0],
                      shared_up=sh[1], shared_down=sh[2])


def build_x(cfg, attempts=None, layer: int = 0, device="cuda", T=None):
    """Activations [T][D] (bf16 bits as int16, or fp32) on the device."""
    T = cfg.T if T is None else T
    dev = torch.device(device)
    att = None if attempts is None else torch.as_tensor(attempts, dtype=torch.int32, device=dev)
    if cfg.x_dtype == "bf16":
        x = torch.empty((T, cfg.D), dtype=torch.int16, device=dev)
        dsgen.dev_x(cfg, None, x, att, layer, T)
    else:
        x = torch.empty((T, cfg.D), dtype=torch.float32, device=dev)
        dsgen.dev_x(cfg, x, None, att, layer, T)
    return x
