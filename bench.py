"""Benchmark of the routed-MoE layer with Q2_K experts on GB300.

Headline workload: one DeepSeek-V4-Flash-shaped layer, decode batch 1
(x[1,4096] bf16, 256 Q2_K experts of 4096->2048->4096, top-6, bf16 shared
expert of width 2048).  One step = one full layer (router, selection, route,
routed and shared SwiGLU experts, combine) over one token.  Inputs larger
than L2: the timed steps rotate over independently generated layers, as a
decode pass does, so no step finds the previous step's weights in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--layers R] [--no-extra] [--no-cpu-baseline]
                    [--workload prefill|prefill_zipf|decode32|stack|decode_q4k|prefill_small]

Prints one JSON line (rank 0).  Its "extra" object times the metric's other
workloads (prefill T=4096 uniform and Zipf against the bf16 tensor roofline;
decode T=32 Zipf, decode T=1 with Q4_K experts and the 43-layer stack at T=8
against HBM).  --impl reference times the fp64 CPU oracle on a bounded sample
of the decode workload instead; --workload times one other workload alone
(profiling runs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, os.path.join(ROOT, "gen")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import dsgen  # noqa: E402

METRIC = "MoE-layer tokens/s, decode B=1/32 & prefill 4096; % of HBM / bf16 roofline"
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFS = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": HBM_FALLBACK_GBS, "bf16_tflops": BF16_FALLBACK_TFS}, "fallback"


def algorithmic_bytes(cfg, n_experts_used: int, T: int) -> int:
    """Bytes the layer must move: each used expert once, the shared expert,
    the router, x in and out."""
    shared = 3 * cfg.Fs * cfg.D * 2
    router = cfg.E * cfg.D * (2 if cfg.router_dtype == "bf16" else 4)
    xio = T * cfg.D * (2 if cfg.x_dtype == "bf16" else 4) + T * cfg.D * 4
    return n_experts_used * cfg.expert_bytes + shared + router + xio


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm --

def replica_throughput(ms_local: float, steps: int, tokens_per_step: int, world: int, device):
    """Whole-job (ms, tokens/s) of `world` independent replicas that each ran
    `steps` steps of tokens_per_step tokens in ms_local: the job takes as long
    as its slowest replica (max over ranks), and every replica's tokens count.
    With world > 1 the process group must be initialised (nccl with a CUDA
    device, gloo with the CPU)."""
    import torch
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * steps * tokens_per_step / (ms_max / 1e3)


def gpu_arm(args, rank, world, local_rank):
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import build as libbuild
    from bit_quantized_routed_router_gb300 import synthetic

    if rank == 0 or not os.path.exists(ds.LIB_PATH):
        libbuild.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = dsgen.DECODE1
    sh = synthetic.shape_of(cfg)
    R = args.layers
    layers = [synthetic.build_layer(cfg, layer=r, device=dev) for r in range(R)]
    xs = [synthetic.build_x(cfg, layer=r, device=dev) for r in range(R)]
    out = torch.empty((1, cfg.D), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.workspace_bytes(sh, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream

    # used experts per layer (for the algorithmic bytes): read back the route once
    n_used = []
    for r in range(R):
        counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
        ds.layer(sh, layers[r], xs[r], out, ws, debug={"counts": counts}, stream=s)
        n_used.append(int((counts > 0).sum().item()))
    ds.sync_status(s)
    bytes_per_step = statistics.mean(algorithmic_bytes(cfg, u, 1) for u in n_used)

    def step(i):
        r = i % R
        ds.layer(sh, layers[r], xs[r], out, ws, stream=s)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # eager: one ds_moe_layer call per step from Python (host enqueue included)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = min(args.steps, 400)
    ev0.record(stream)
    for i in range(n_eager):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms_per_step = ev0.elapsed_time(ev1) / n_eager
    # timed: the same ds_moe_layer calls captured once into a CUDA graph of
    # gsteps steps (cycling the layers) and replayed, so that the host's
    # enqueue cost does not decide the number; the remainder runs eagerly
    gsteps = min(args.steps, 10 * R)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(gsteps):
            ds.layer(sh, layers[i % R], xs[i % R], out, ws)
    reps, rem = divmod(args.steps, gsteps)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    clocks = Clocks(local_rank)
    if world > 1:
        torch.distributed.barrier()
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(reps):
        graph.replay()
    for i in range(rem):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ds.sync_status(s)
    ms_max, value = replica_throughput(ms, args.steps, cfg.T, world, dev)
    ms_per_step = ms_max / args.steps

    # end to end through the host-buffer entry point: x H2D, layer, out D2H per step
    xh = [x.cpu().pin_memory() for x in xs]
    oh = torch.empty((1, cfg.D), dtype=torch.float32).pin_memory()
    ws_h = torch.empty(ds.workspace_bytes(sh, 1), dtype=torch.uint8, device=dev)
    for i in range(args.warmup):
        ds.layer_hostio(sh, layers[i % R], xh[i % R], oh, ws_h, stream=s)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        ds.layer_hostio(sh, layers[i % R], xh[i % R], oh, ws_h, stream=s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    _, e2e_value = replica_throughput(e2e_ms, args.steps, cfg.T, world, dev)

    pk, pk_kind = peaks()
    hbm = float(pk.get("hbm_gbs", HBM_FALLBACK_GBS))
    achieved = bytes_per_step / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox generator; weights N(0,0.02) packed to Q2_K)",
        "config": {"workload": cfg.name, "T": cfg.T, "n_embd": cfg.D, "n_expert": cfg.E,
                   "top_k": cfg.k, "n_ff": cfg.F, "n_ff_shared": cfg.Fs,
                   "expert_format": "Q2_K 84 B / 256 weights", "shared_dtype": "bf16",
                   "l2": f"inputs larger than L2: steps rotate over {R} independently generated "
                         f"layers ({R * (cfg.E * cfg.expert_bytes) / 1e9:.1f} GB of experts)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": f"CUDA graph of {gsteps} ds_moe_layer calls replayed {reps}x "
                             f"(+{rem} eager); eager Python calls: {eager_ms_per_step * 1e3:.1f} us/step"},
        "roofline": {"bound": "hbm", "kernel": "decode step: route_kernel + stream_kernel (both timed as one launch)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": pk_kind,
                     "traffic": DECODE_STEP_DRAM_BYTES, "algorithmic_bytes": bytes_per_step},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": cfg.T * cfg.D * 2,
                "d2h_bytes_per_step": cfg.T * cfg.D * 4},
        "gpu_launches": args.steps * LAUNCHES_PER_DECODE_STEP,
        "clocks": clk,
    }
    return line


LAUNCHES_PER_DECODE_STEP = 2  # router logits; the one-token streaming kernel
# DRAM bytes read + written by one decode step, from one ncu capture of these
# kernels as they stand (route_kernel 2,118,912 read; stream_kernel
# 100,054,016 read + 3,266,816 written; the commands are in the decode profile
# summary).  Set to None whenever either kernel changes until it is captured
# again.
DECODE_STEP_DRAM_BYTES = 105_439_744

PREFILL_FLOPS = 1.4517e12  # 4096 x (6*3*2*D*F + 3*2*D*F + 2*D*E) at the Flash shape


def time_layer(cfg, iters, dev, warmup=3):
    """(ms per layer call, used experts, path) for one synthetic layer of cfg
    with its inputs resident; CUDA events over `iters` calls after warm-up."""
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import synthetic

    sh = synthetic.shape_of(cfg)
    W = synthetic.build_layer(cfg, device=dev)
    x = synthetic.build_x(cfg, device=dev)
    out = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    ds.layer(sh, W, x, out, ws, debug={"counts": counts})
    used = int((counts > 0).sum().item())
    for _ in range(warmup):
        ds.layer(sh, W, x, out, ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        ds.layer(sh, W, x, out, ws)
    e1.record()
    torch.cuda.synchronize(dev)
    ds.sync_status()
    path = ds.layer_path(sh, cfg.T, x)
    del W, ws, out
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / iters, used, path


def time_decode_rotating(cfg, R, iters, dev, warmup=3):
    """(ms per one-token layer call, mean used experts, path) with the calls
    rotating over R independently generated layers (so that one call's
    experts are not in L2 from the previous one), captured into a CUDA graph
    of 10 R calls and replayed."""
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import synthetic

    sh = synthetic.shape_of(cfg)
    layers = [synthetic.build_layer(cfg, layer=r, device=dev) for r in range(R)]
    xs = [synthetic.build_x(cfg, layer=r, device=dev) for r in range(R)]
    out = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    used = []
    for r in range(R):
        ds.layer(sh, layers[r], xs[r], out, ws, debug={"counts": counts})
        used.append(int((counts > 0).sum().item()))
    for i in range(warmup):
        ds.layer(sh, layers[i % R], xs[i % R], out, ws)
    torch.cuda.synchronize(dev)
    g = 10 * R
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(g):
            ds.layer(sh, layers[i % R], xs[i % R], out, ws)
    graph.replay()
    torch.cuda.synchronize(dev)
    reps = max(1, iters // g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ds.sync_status()
    path = ds.layer_path(sh, cfg.T, xs[0])
    del layers, ws, out
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / (reps * g), statistics.mean(used), path


def time_stack(cfg, iters, dev, warmup=3):
    """The 43-layer stack (x += layer(bf16(RMSNorm(x))) per layer, T tokens):
    (ms per step, bytes read per step, distinct experts per layer, path).  One
    step = the residual reset to the same input (a 128 KB device copy) + one
    ds_moe_stack call over every layer, all experts resident, captured once
    into a CUDA graph and replayed.  The experts a
    step reads are counted on an untimed pass that advances the same residual
    one layer at a time (bit-identical to the multi-layer call) and reads each
    layer's expert counts from a ds_moe_layer call on the normalised input."""
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import synthetic
    from dataclasses import replace

    sh = synthetic.shape_of(cfg)
    Ws = [synthetic.build_layer(cfg, l, device=dev) for l in range(cfg.layers)]
    x0 = torch.from_numpy(dsgen.host_x(replace(cfg, x_dtype="f32"))).to(dev)
    x = x0.clone()
    ws = torch.empty(ds.workspace_bytes(sh, cfg.T), dtype=torch.uint8, device=dev)
    out = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    used = []
    for W in Ws:
        xn = (x * torch.rsqrt(x.square().mean(dim=1, keepdim=True) + 1e-6)).to(torch.bfloat16)
        ds.layer(sh, W, xn, out, ws, debug={"counts": counts})
        used.append(int((counts > 0).sum().item()))
        ds.stack(sh, [W], x, ws)
    ds.sync_status()
    for _ in range(warmup):
        x.copy_(x0)
        ds.stack(sh, Ws, x, ws)
    torch.cuda.synchronize(dev)
    # the step (residual reset + one ds_moe_stack call, 8 launches per layer)
    # captured once into a CUDA graph and replayed
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        x.copy_(x0)
        ds.stack(sh, Ws, x, ws)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ds.sync_status()
    path = ds.layer_path(sh, cfg.T, xn)
    per_layer_fixed = cfg.Fs * cfg.D * 2 * 3 + cfg.E * cfg.D * 2
    b = sum(u * cfg.expert_bytes + per_layer_fixed for u in used)
    del Ws, ws, out, x, x0
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / iters, b, used, path


def time_resident(cfg, R, budgets, n_tokens, dev):
    """One-token decode with the routed experts of R layers in pinned host
    memory and a device cache (ds_moe_cache_layer) holding a fraction of
    them: per budget, ms per layer call (wall clock: every call reads back
    its route to update the cache), the hit rate and the bytes the calls
    read from host memory.  One warm-up pass of n_tokens tokens through the
    R layers, then one timed pass of other tokens."""
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import synthetic
    from dataclasses import replace

    sh = synthetic.shape_of(cfg)
    eb = cfg.expert_bytes
    Ws, hosts = [], []
    for r in range(R):
        W = synthetic.build_layer(cfg, layer=r, device=dev)
        h = torch.empty(W.experts.shape, dtype=W.experts.dtype, pin_memory=True)
        h.copy_(W.experts)
        hosts.append(h)
        Ws.append(replace(W, experts=None))  # the device copy is dropped
        del W
    torch.cuda.empty_cache()
    ws = torch.empty(ds.workspace_bytes(sh, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((1, cfg.D), dtype=torch.float32, device=dev)
    res = {}
    for frac in budgets:
        n_slots = int(round(frac * R * cfg.E))
        slots = torch.empty((max(n_slots, 1), eb), dtype=torch.uint8, device=dev)
        tables = torch.empty((R, cfg.E), dtype=torch.int32, device=dev)
        c = ds.ExpertCache(sh, hosts, slots, n_slots, tables)
        for t in range(n_tokens):
            x = synthetic.build_x(cfg, layer=1000 + t, device=dev)
            for r in range(R):
                c.layer(r, Ws[r], x, out, ws)
        xs = [synthetic.build_x(cfg, layer=2000 + t, device=dev) for t in range(n_tokens)]
        ds.sync_status()
        st0 = c.stats()
        torch.cuda.synchronize(dev)
        calls = []
        t0 = time.perf_counter()
        for t in range(n_tokens):
            for r in range(R):
                t1 = time.perf_counter()
                c.layer(r, Ws[r], xs[t], out, ws)  # synchronous: it reads back the route
                calls.append(time.perf_counter() - t1)
        torch.cuda.synchronize(dev)
        ms = (time.perf_counter() - t0) * 1e3 / (n_tokens * R)
        ds.sync_status()
        st1 = c.stats()
        hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
        calls.sort()
        res[f"{frac:g}"] = {"slots": n_slots, "cache_gb": n_slots * eb / 1e9, "ms_per_layer": ms,
                            "median_ms_per_call": calls[len(calls) // 2] * 1e3,
                            "max_ms_per_call": calls[-1] * 1e3,
                            "tokens_per_s_per_layer": 1e3 / ms, "hit_rate": hits / max(1, hits + misses),
                            "host_expert_bytes_per_call": misses * eb / (n_tokens * R)}
        c.close()
        del slots, tables
        torch.cuda.empty_cache()
    del Ws, hosts, ws, out
    return res


def extra_workloads(args, dev):
    """The other timed workloads of the metric (not the headline line):
    prefill T=4096 (uniform and Zipf router) against the bf16 tensor roofline,
    decode T=32 Zipf, decode T=1 with Q4_K experts and the 43-layer stack at
    T=8 against the HBM roofline.  Each on its own layer, inputs
    resident, CUDA events over `iters` layer calls after warm-up."""
    import torch
    import bit_quantized_routed_router_gb300 as ds
    from bit_quantized_routed_router_gb300 import synthetic

    pk, pk_kind = peaks()
    res = {}
    for cfg, iters in ((dsgen.PREFILL, 10), (dsgen.PREFILL_ZIPF, 10), (PREFILL_Q4K, 10),
                       (dsgen.DECODE32_ZIPF, 200)):
        if cfg.T < 64:  # decode-sized: rotate four layers (inputs larger than L2), graph-timed
            ms, used, path = time_decode_rotating(cfg, 4, iters, dev)
        else:
            ms, used, path = time_layer(cfg, iters, dev)
        entry = {"tokens_per_s": cfg.T / (ms / 1e3), "ms_per_layer": ms, "T": cfg.T,
                 "used_experts": used, "path": path}
        if cfg.T >= 64:
            tfs = PREFILL_FLOPS / (ms / 1e3) / 1e12
            peak = float(pk.get("bf16_tflops", BF16_FALLBACK_TFS))
            entry["roofline"] = {"bound": "tensor", "achieved": tfs, "peak": peak, "unit": "TFLOP/s",
                                 "frac": tfs / peak, "peak_source": pk_kind,
                                 "algorithmic_flops": PREFILL_FLOPS}
        else:
            b = algorithmic_bytes(cfg, used, cfg.T)
            gbs = b / (ms / 1e3) / 1e9
            hbm = float(pk.get("hbm_gbs", HBM_FALLBACK_GBS))
            entry["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                 "frac": gbs / hbm, "peak_source": pk_kind, "algorithmic_bytes": b}
            entry["timing"] = "CUDA graph of 40 calls rotating over 4 layers"
        res[cfg.name] = entry
    cfg = dsgen.DECODE1_Q4K
    ms, used, path = time_decode_rotating(cfg, 2, 400, dev)
    b = algorithmic_bytes(cfg, used, cfg.T)
    gbs = b / (ms / 1e3) / 1e9
    hbm = float(pk.get("hbm_gbs", HBM_FALLBACK_GBS))
    res[cfg.name] = {"tokens_per_s": cfg.T / (ms / 1e3), "ms_per_layer": ms, "T": cfg.T,
                     "used_experts": used, "path": path,
                     "timing": "CUDA graph of 20 calls rotating over 2 layers",
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                  "frac": gbs / hbm, "peak_source": pk_kind, "algorithmic_bytes": b}}
    cfg = RESIDENT
    res[cfg.name] = {"T": 1, "layers": 2, "budgets": time_resident(cfg, 2, (0.0, 0.25, 1.0), 24, dev),
                     "timing": "wall clock per ds_moe_cache_layer call (each reads back its route); "
                               "budget = fraction of the layers' experts that fit in device slots",
                     "experts": "routed experts in pinned host memory, read in place when not cached"}
    cfg = dsgen.STACK
    ms, b, used, path = time_stack(cfg, 20, dev)
    gbs = b / (ms / 1e3) / 1e9
    hbm = float(pk.get("hbm_gbs", HBM_FALLBACK_GBS))
    res[cfg.name] = {"tokens_per_s": cfg.T / (ms / 1e3), "ms_per_step": ms, "T": cfg.T,
                     "layers": cfg.layers, "bytes_read_per_s": b / (ms / 1e3),
                     "used_experts_per_layer": {"min": min(used), "max": max(used),
                                                "mean": sum(used) / len(used)},
                     "path": path,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                  "frac": gbs / hbm, "peak_source": pk_kind, "algorithmic_bytes": b}}
    return res


PREFILL_Q4K = replace(dsgen.PREFILL, name="prefill T=4096 Q4_K experts D=4096 E=256 k=6 F=2048 Fs=2048",
                      expert_fmt="q4k")
DECODE8 = replace(dsgen.DECODE1, name="decode T=8 D=4096 E=256 k=6 F=2048 Fs=2048 (one layer)", T=8)
RESIDENT = replace(dsgen.DECODE1, name="decode T=1 experts in host memory, device cache, zipf(1.1) "
                                       "D=4096 E=256 k=6 F=2048 Fs=2048", zipf_s=1.1)

# single workloads for profiling runs (not the benchmark line)
WORKLOADS = {
    "prefill": dsgen.PREFILL,
    "prefill_zipf": dsgen.PREFILL_ZIPF,
    "decode32": dsgen.DECODE32_ZIPF,
    "decode8": DECODE8,
    "stack": dsgen.STACK,
    "decode_q4k": dsgen.DECODE1_Q4K,
    "prefill_q4k": PREFILL_Q4K,
    "resident": RESIDENT,
    # same shapes at 1/4 of the experts and tokens (about 96 tokens per
    # expert as at full size): a case small enough for full profiler captures
    "prefill_small": None,
}


# ------------------------------------------------------------ oracle (CPU) --

def host_info():
    """The host's logical core count and CPU model (for the CPU-baseline rows)."""
    model = None
    impl_arm = False
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k = k.strip().lower()
                if k in ("model name", "cpu model", "hardware") and v.strip():
                    model = v.strip()
                    break
                if k == "cpu implementer" and v.strip() == "0x41":
                    impl_arm = True
                if k == "cpu part" and model is None:
                    # Arm's published part numbers for the cores these hosts use
                    part = v.strip().lower()
                    names = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
                             "0xd49": "Arm Neoverse N2", "0xd84": "Arm Neoverse V3"}
                    model = names.get(part, f"Arm cpu part {part}") if impl_arm else f"cpu part {part}"
    except OSError:
        pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return {"host_cores": os.cpu_count() or 1, "cpu_model": model}


def oracle_sample(n_tokens: int = 2, budget_s: float = 12.0):
    """Time the fp64 oracle on decode-B=1 steps (one token each) of the same
    layer shape.  The experts the sampled tokens select are regenerated and
    packed once (input preparation, untimed); then whole layer evaluations
    (router, selection, routed and shared experts, combine) of those tokens
    are timed in turn until about budget_s seconds of compute.  `cores` is
    the number of threads the oracle's work split used (one per selected
    expert plus the shared expert, at most the host's cores)."""
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import oracle

    cfg = dsgen.DECODE1
    lo = oracle.LayerOracle(cfg)
    xs, exps = [], []
    for t in range(n_tokens):
        x = oracle.as_f64(dsgen.host_x(cfg, [t])[:1], cfg.x_dtype)
        ids0, _ = oracle.select(lo.logits(x), cfg.k)
        xs.append(x)
        exps.append(lo.experts(ids0))
    times, used_threads = [], 0
    while sum(times) < budget_s or len(times) < n_tokens:
        i = len(times) % n_tokens
        t0 = time.perf_counter()
        L = lo.logits(xs[i])
        ids, w = oracle.select(L, cfg.k)
        oracle.moe_layer(xs[i], exps[i], lo.shared, ids, w, cfg.D, cfg.E, cfg.F, cfg.Fs,
                         fmt=cfg.expert_fmt)
        times.append(time.perf_counter() - t0)
        used_threads = max(used_threads, min(oracle.NTHREADS, len(set(ids.ravel())) + 1))
    tot = sum(times)
    return {"value": len(times) / tot, "unit": "tokens/s", "cores": used_threads,
            "kind": "oracle", **host_info(),
            "sample": f"{len(times)} decode-B=1 layer evaluations cycling over {n_tokens} seeded "
                      f"tokens of the same layer (fp64 C oracle, {tot:.1f} s of layer compute; "
                      f"expert regeneration untimed)"}


def oracle_batch_sample(cfg, n_tokens: int, what: str):
    """The fp64 oracle on one layer evaluation of the first n_tokens tokens of
    a batched workload (decode T=32, prefill, a stack layer): tokens/s of
    that evaluation; the selected experts are regenerated first (untimed)."""
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import oracle
    from dataclasses import replace

    c = replace(cfg, T=n_tokens)
    lo = oracle.LayerOracle(c)
    x = oracle.as_f64(dsgen.host_x(c), c.x_dtype)
    ids0, _ = oracle.select(lo.logits(x), c.k)
    exps = lo.experts(ids0)
    t0 = time.perf_counter()
    L = lo.logits(x)
    ids, w = oracle.select(L, c.k)
    oracle.moe_layer(x, exps, lo.shared, ids, w, c.D, c.E, c.F, c.Fs, fmt=c.expert_fmt)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": min(oracle.NTHREADS, len(exps) + 1),
            "kind": "oracle", **host_info(),
            "sample": f"one layer evaluation of {n_tokens} tokens of the {what} workload "
                      f"({len(exps)} experts, fp64 C oracle, {dt:.1f} s; expert regeneration untimed)"}


def reference_arm(args, rank):
    if rank != 0:
        return None
    cb = oracle_sample(2, budget_s=min(60.0, max(5.0, 0.5 * args.steps)))
    cfg = dsgen.DECODE1
    return {"metric": METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / cb["value"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox generator)", "impl": "reference",
            "config": {"workload": cfg.name, "T": 1},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=4, help="rotating layers (L2 defeat)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill / decode-32 extras")
    ap.add_argument("--workload", default="decode", choices=["decode"] + list(WORKLOADS),
                    help="time one other workload only (profiling runs); prints its own JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.workload != "decode":
        import torch
        from dataclasses import replace
        from bit_quantized_routed_router_gb300 import build as libbuild
        libbuild.build()
        cfg = WORKLOADS[args.workload] or replace(dsgen.PREFILL, name="prefill T=1024 E=64 (profiling case)",
                                                   T=1024, E=64)
        if args.workload == "decode_q4k":
            ms, used, path = time_decode_rotating(cfg, 2, args.steps, torch.device("cuda", 0),
                                                  warmup=args.warmup)
            print(json.dumps({"workload": cfg.name, "ms_per_layer": ms, "tokens_per_s": cfg.T / (ms / 1e3),
                              "used_experts": used, "path": path, "steps": args.steps}), flush=True)
            return
        if args.workload == "resident":
            r = time_resident(cfg, 2, (0.0, 0.25, 1.0), max(2, args.steps), torch.device("cuda", 0))
            print(json.dumps({"workload": cfg.name, "budgets": r}), flush=True)
            return
        if args.workload == "stack":
            ms, b, used, path = time_stack(cfg, args.steps, torch.device("cuda", 0), warmup=args.warmup)
            print(json.dumps({"workload": cfg.name, "ms_per_step": ms, "tokens_per_s": cfg.T / (ms / 1e3),
                              "bytes_read_per_s": b / (ms / 1e3), "used_experts": used, "path": path,
                              "steps": args.steps}), flush=True)
            return
        ms, used, path = time_layer(cfg, args.steps, torch.device("cuda", 0), warmup=args.warmup)
        print(json.dumps({"workload": cfg.name, "ms_per_layer": ms, "tokens_per_s": cfg.T / (ms / 1e3),
                          "used_experts": used, "path": path, "steps": args.steps}), flush=True)
        return

    if args.impl == "reference":
        line = reference_arm(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = gpu_arm(args, rank, world, local_rank)
    if rank == 0 and not args.no_extra and world == 1:
        import torch
        line["extra"] = extra_workloads(args, torch.device("cuda", local_rank))
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_sample()
            if "extra" in line:
                for cfg, n, what in ((dsgen.DECODE32_ZIPF, 32, "decode T=32 Zipf"),
                                     (dsgen.PREFILL, 8, "prefill T=4096 (a sample of its tokens)"),
                                     (dsgen.STACK, 8, "43-layer stack (its first layer)")):
                    if cfg.name in line["extra"]:
                        line["extra"][cfg.name]["cpu_baseline"] = oracle_batch_sample(cfg, n, what)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
