#!/usr/bin/env python
"""Benchmark of the NVFP4 routed-expert MoE layer step on GB300.

One step = one moe_nvfp4_layer call (route-group, gather+quantize, grouped
GEMM w13, SwiGLU+requantize, grouped GEMM w2, scatter-add) over one batch of
synthetic input already resident in HBM, timed with CUDA events on its stream
as a direct call (`--graph`: as a CUDA-graph replay of that call; the other
way is reported beside it). The L2 is flushed (a write of twice its size,
then a read of another buffer) before every timed step and the routing
rotates over 20 seeded draws, so weights always stream from HBM.

Prints one JSON line. value = weight-stream GB/s: algorithmic bytes per step
(active experts' packed weights + block scales, x, y, routing, globals) over
the mean device time of a step. `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer ms/step and weight-stream GB/s (% of HBM roofline) at M=1/8/32"
FALLBACK_HBM_GBS = 6800.0
N_ROUTINGS = 20
# the GEMM kernel's source: its translation unit and the headers it includes
GEMM_SRC = [os.path.join(ROOT, "nvfp4_block_scaled_gather_gb300", "csrc", f)
            for f in ("nvfp4_gemm.cu", "nvfp4_codec.cuh", "ldcg.cuh", "pdl.cuh", "internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "expert_gemms_decode_m1_traffic.txt")


def expert_bytes(H, I):
    """Packed e2m1 + e4m3 block scales of one expert: w13 2I x H, w2 H x I."""
    return 3 * H * I * 9 // 16


def step_bytes(cfg, G, T):
    """Algorithmic bytes of one layer step: active experts' weights, x read,
    y written, routing ids + weights, per-expert globals."""
    return G * expert_bytes(cfg.H, cfg.I) + 2 * T * cfg.H * 2 + T * cfg.k * 8 + 12 * cfg.E


def gemms_launch_bytes(cfg, G, R):
    """Algorithmic bytes of the layer's GEMM launch (w13 with SwiGLU and
    requantization in its epilogue, then w2): the active experts' w13 and w2
    (e2m1 + scales), the NVFP4 token rows and scales read, the NVFP4 h rows
    and scales written and read back, the fp32 d2 rows written."""
    return G * expert_bytes(cfg.H, cfg.I) + R * cfg.H * 9 // 16 + 2 * (R * cfg.I * 9 // 16) + R * cfg.H * 4


def max_over_ranks(value, dist_mod, device):
    """The largest of every rank's value (a replica run's time is its slowest
    rank's); the value itself when not distributed."""
    if not dist_mod:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, bytes_per_rank, total_ms):
    """Whole-job GB/s of `world` replicas that each moved bytes_per_rank in
    the slowest rank's total_ms."""
    return world * bytes_per_rank / (total_ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm"):
            if key in d:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def gemm_source_sha() -> str:
    """First 16 hex digits of the SHA-256 of the GEMM kernel's source files, in order."""
    h = hashlib.sha256()
    for path in GEMM_SRC:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """ncu DRAM bytes per GEMM launch (decode M=1), if recorded for the
    current kernel source; None when absent or when the kernel changed since."""
    try:
        sha = gemm_source_sha()
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    a, b = line.split(":", 1)
                    kv[a.strip()] = b.strip()
        if kv.get("kernel_source_sha256_16") == sha:
            return int(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def wait_first(self):
        """Blocks until nvidia-smi printed its first sample (or exited)."""
        self._first = self.proc.stdout.readline() if self.proc else None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        lines = [ln for ln in ((self._first or "") + out).splitlines() if ln.strip()]
        sm, mx, reasons = [], 0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, parts[2:]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gpu_bench(args, rank, world):
    import torch

    from nvfp4_block_scaled_gather_gb300 import _native as N
    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_activations, make_routing, make_weights

    import dataclasses
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)
    N.load()

    cfg = CONFIGS[args.config]
    if args.experts:
        cfg = dataclasses.replace(cfg, E=args.experts)
    w = make_weights(cfg.E, cfg.H, cfg.I, device=dev)
    W = N.Weights(w["w13_packed"], w["w13_sf_linear"], w["g_gate_up"], w["w2_packed"], w["w2_sf_linear"],
                  w["g_down"])
    del w
    flush = torch.empty(2 * props.L2_cache_size, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(2 * props.L2_cache_size // 4, dtype=torch.int32, device=dev)

    def workload(c, n=N_ROUTINGS):
        items = []
        for i in range(n):
            ids, tw = make_routing(c, seed=2 + 1000 * i)
            T = ids.shape[0]
            x = make_activations(T, c.H, seed=1 + 1000 * i, device=dev)
            valid = ids[(ids >= 0) & (ids < c.E)]
            G = int(torch.unique(valid).numel())
            items.append(dict(x=x, ids=ids.to(dev), tw=tw.to(dev), ids_h=ids, tw_h=tw, T=T, G=G,
                              R=int(valid.numel())))
        return items

    def flush_l2():
        """Write a buffer twice the L2, then read another: the weights leave
        L2 and the lines left behind are clean (no write-backs in the step)."""
        flush.zero_()
        flush_read.sum(dtype=torch.int32)

    warm_cache = {}

    def code_warmer(c, T):
        """A tiny layer step (8 experts, hidden 256, intermediate 128, weights
        of its own) taking the same kernel paths as a step of T tokens of
        config c: run after the L2 flush, untimed, it brings the kernels'
        code back into L2 and leaves the timed step's weights, activations
        and routing cold -- the state of a model whose every layer runs these
        kernels with its own weights."""
        S = T * c.k
        lay = N.layer_sf_layout(T, c.k, c.E)
        Tw = 1 if S <= 32 else (16 if lay == N.SF_ATOM128 else 8)
        if Tw not in warm_cache:
            tw_cfg = dataclasses.replace(CONFIGS["tiny"], E=8, k=8, T=Tw)
            w8 = make_weights(8, 256, 128, seed=77, device=dev)
            W8 = N.Weights(w8["w13_packed"], w8["w13_sf_linear"], w8["g_gate_up"], w8["w2_packed"],
                           w8["w2_sf_linear"], w8["g_down"])
            ids8, tw8 = make_routing(tw_cfg, seed=77)
            x8 = make_activations(Tw, 256, seed=77, device=dev)
            y8 = torch.empty_like(x8)
            lay8 = N.MoeLayer(W8, Tw, 8)
            assert N.layer_sf_layout(Tw, 8, 8) == lay
            ids8, tw8 = ids8.to(dev), tw8.to(dev)
            warm_cache[Tw] = (lay8.capture(x8, ids8, tw8, y8), W8, x8, ids8, tw8, y8, lay8)
        return warm_cache[Tw][0]

    def time_layer(c, items, steps, warmup, sampler=None, graph=False, code_warm=False):
        """Times `steps` layer steps (mean and per-step CUDA events), L2
        flushed before each. graph=True replays one CUDA graph per routing
        (captured from the same C-ABI call); graph=False calls it directly.
        code_warm: after each flush, a tiny untimed step through the same
        kernels (code_warmer) so their code is in L2 and only the data is
        cold."""
        T_max = max(it["T"] for it in items)
        warm = code_warmer(c, T_max) if code_warm else None
        layer = N.MoeLayer(W, T_max, c.k)
        ys = [torch.empty_like(it["x"]) for it in items]
        if graph:
            graphs = [layer.capture(it["x"], it["ids"], it["tw"], y) for it, y in zip(items, ys)]
            run = lambda i: graphs[i % len(items)].replay()  # noqa: E731
        else:
            def run(i):
                it = items[i % len(items)]
                layer(it["x"], it["ids"], it["tw"], ys[i % len(items)])
        for i in range(warmup):
            run(i)
        if sampler is not None:
            # keep the clocks sampler busy for at least ~1 s of load before timing
            t0 = time.time()
            i = 0
            while time.time() - t0 < 1.0:
                flush_l2()
                run(i)
                i += 1
                if i % 20 == 0:
                    torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            flush_l2()
            if warm is not None:
                warm.replay()
            ev[i][0].record(stream)
            run(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ms = [a.elapsed_time(b) for a, b in ev]
        byts = [step_bytes(c, items[i % len(items)]["G"], items[i % len(items)]["T"]) for i in range(steps)]
        return ms, byts

    def time_w4a16(c, items, steps):
        """The GEMV path (W4A16) of the same step, graph replays, L2 flushed
        before each: a validation path, timed for the record."""
        T_max = max(it["T"] for it in items)
        layer = N.MoeLayerW4A16(W, T_max, c.k)
        ys = [torch.empty_like(it["x"]) for it in items]
        graphs = [layer.capture(it["x"], it["ids"], it["tw"], y) for it, y in zip(items, ys)]
        for i in range(3):
            graphs[i % len(items)].replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            flush_l2()
            ev[i][0].record(stream)
            graphs[i % len(items)].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in ev]
        byts = [step_bytes(c, items[i % len(items)]["G"], items[i % len(items)]["T"]) for i in range(steps)]
        return ms, byts

    def time_stages(c, items, steps):
        """The step through the separate entry points, stage by stage with
        events between them: route, gather + quantize by rows, the two-GEMM
        launch (the layer's own GEMM kernel and token blocks), scatter. The
        layer itself routes and quantizes in one launch for decode batches and
        quantizes token by token otherwise."""
        T_max = max(it["T"] for it in items)
        S = T_max * c.k
        lay = N.layer_sf_layout(T_max, c.k, c.E)  # the token blocks the layer itself takes
        G_ = N.Groups(T_max, c.k, c.E, dev)
        xq = torch.empty(S, c.H // 2, dtype=torch.uint8, device=dev)
        xsf = torch.empty(N.sf_bytes(S, c.E, c.H, lay), dtype=torch.uint8, device=dev)
        hq = torch.empty(S, c.I // 2, dtype=torch.uint8, device=dev)
        hsf = torch.empty(N.sf_bytes(S, c.E, c.I, lay), dtype=torch.uint8, device=dev)
        d2 = torch.empty(S, c.H, dtype=torch.float32, device=dev)
        gate = torch.zeros(N.expert_gemms_gate_bytes(S, c.E, c.I), dtype=torch.uint8, device=dev)  # zeroed once
        names = ["route", "gather_quantize", "expert_gemms", "scatter"]
        acc = {n: [] for n in names}
        gemm_bytes = []
        for i in range(steps + 3):
            it = items[i % len(items)]
            T = it["T"]
            G1 = N.Groups(T, c.k, c.E, dev) if T != T_max else G_
            y = torch.empty_like(it["x"])
            flush_l2()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
            evs[0].record(stream)
            N.moe_route_groups(it["ids"], c.E, G1)
            evs[1].record(stream)
            N.moe_gather_quantize_rows(it["x"], c.k, G1, xq, xsf, lay)
            evs[2].record(stream)
            N.nvfp4_moe_expert_gemms(xq, xsf, G1, W, hq, hsf, d2, gate, layout=lay)
            evs[3].record(stream)
            N.moe_scatter_add(d2, it["ids"], it["tw"], c.E, G1, W.g_down, y)
            evs[4].record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                for j, n in enumerate(names):
                    acc[n].append(evs[j].elapsed_time(evs[j + 1]))
                gemm_bytes.append(gemms_launch_bytes(c, it["G"], it["R"]))
        return {n: statistics.mean(v) for n, v in acc.items()}, statistics.mean(gemm_bytes)

    def time_e2e(c, items, steps, graph=False):
        """Through the public call with host buffers: one pinned H2D copy of the
        step's inputs (x, ids and router weights packed in one staging buffer,
        whose device twin the layer reads in place), the layer step (the call,
        or its captured graph), D2H of y; all inside the timed region, which
        like the other timings opens on the stream right after the L2 flush
        (the host has queued the step's work by then)."""
        T_max = max(it["T"] for it in items)
        layer = N.MoeLayer(W, T_max, c.k)

        def carve(buf, it):
            # x | ids | tw, each section 256-byte aligned
            T, k = it["T"], c.k
            nx, ni = T * c.H * 2, T * k * 4
            ox, oi, ow = 0, (nx + 255) // 256 * 256, 0
            ow = oi + (ni + 255) // 256 * 256
            x = buf[ox:ox + nx].view(torch.bfloat16).view(T, c.H)
            ids = buf[oi:oi + ni].view(torch.int32).view(T, k)
            tw = buf[ow:ow + ni].view(torch.float32).view(T, k)
            return x, ids, tw, ow + ni

        host, dev_bufs, graphs = [], [], []
        for it in items:
            size = carve(torch.empty(1 << 30, dtype=torch.uint8, device="meta"), it)[3]
            hbuf = torch.empty(size, dtype=torch.uint8).pin_memory()
            hx, hi, hw, _ = carve(hbuf, it)
            hx.copy_(it["x"].cpu()), hi.copy_(it["ids_h"]), hw.copy_(it["tw_h"])
            host.append(dict(buf=hbuf, y=torch.empty_like(it["x"], device="cpu").pin_memory(), T=it["T"], G=it["G"]))
            dbuf = torch.empty(size, dtype=torch.uint8, device=dev)
            dx, di, dw, _ = carve(dbuf, it)
            dbuf.copy_(hbuf)
            y = torch.empty_like(it["x"])
            graphs.append(layer.capture(dx, di, dw, y) if graph else None)
            dev_bufs.append(dict(buf=dbuf, y=y, x=dx, ids=di, tw=dw))
        ms, h2d, d2h, byts = [], [], [], []
        for i in range(steps + 3):
            h, d = host[i % len(host)], dev_bufs[i % len(host)]
            torch.cuda.synchronize()
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            d["buf"].copy_(h["buf"], non_blocking=True)
            if graph:
                graphs[i % len(host)].replay()
            else:
                layer(d["x"], d["ids"], d["tw"], d["y"])
            h["y"].copy_(d["y"], non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
                h2d.append(d["buf"].numel())
                d2h.append(d["y"].numel() * 2)
                byts.append(step_bytes(c, h["G"], h["T"]))
        return ms, byts, statistics.mean(h2d), statistics.mean(d2h)

    def time_e2e_zero_copy(c, items, steps):
        """The same public call with its inputs and y in pinned host memory,
        passed as they are: with unified addressing the step's kernels read x,
        the routing and the router weights over the CPU-GPU link and write y
        there, so no separate copy is queued. Checked bit for bit against the
        call on device buffers before timing."""
        T_max = max(it["T"] for it in items)
        layer = N.MoeLayer(W, T_max, c.k)
        host = []
        for it in items:
            hx = it["x"].cpu().pin_memory()
            hi = it["ids_h"].clone().pin_memory()
            hw = it["tw_h"].clone().pin_memory()
            hy = torch.empty_like(hx).pin_memory()
            host.append((hx, hi, hw, hy, it))
        hx, hi, hw, hy, it = host[0]
        want = layer(it["x"], it["ids"], it["tw"]).cpu()
        layer(hx, hi, hw, hy)
        torch.cuda.synchronize()
        assert torch.equal(hy.view(torch.int16), want.view(torch.int16)), "host-buffer call differs"
        ms, byts, h2d, d2h = [], [], [], []
        for i in range(steps + 3):
            hx, hi, hw, hy, it = host[i % len(host)]
            torch.cuda.synchronize()
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            layer(hx, hi, hw, hy)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
                h2d.append(hx.numel() * 2 + hi.numel() * 4 + hw.numel() * 4)
                d2h.append(hy.numel() * 2)
                byts.append(step_bytes(c, it["G"], it["T"]))
        return ms, byts, statistics.mean(h2d), statistics.mean(d2h)

    try:
        gpu_id = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        gpu_id = str(local)
    items = workload(cfg)
    if args.profile:
        # short run for profilers: warm-up, then the timed steps, nothing else
        if args.path == "w4a16":
            ms, byts = time_w4a16(cfg, items, args.steps)
        else:
            ms, byts = time_layer(cfg, items, args.steps, args.warmup, graph=False)
        print(json.dumps({"profile_run": cfg.name, "path": args.path, "experts": cfg.E,
                          "ms_per_step": statistics.mean(ms)}))
        return
    sampler = ClockSampler(gpu_id)
    sampler.wait_first()
    ms, byts = time_layer(cfg, items, args.steps, args.warmup, sampler, graph=args.graph)
    clocks = sampler.stop()
    ms_other, _ = time_layer(cfg, items, max(10, min(args.steps, 40)), 3, graph=not args.graph)
    ms_warm, _ = time_layer(cfg, items, max(10, min(args.steps, 40)), 3, graph=args.graph, code_warm=True)
    total_ms = max_over_ranks(sum(ms), dist, dev)
    ms_step = total_ms / args.steps
    gbs = replica_throughput(world, sum(byts), total_ms)

    stages, gemm_bytes = time_stages(cfg, items, max(5, min(args.steps, 20)))
    peak, peak_kind = measured_peaks()
    achieved = gemm_bytes / (stages["expert_gemms"] * 1e-3) / 1e9
    e2e_ms, e2e_bytes, h2d, d2h = time_e2e(cfg, items, max(5, min(args.steps, 20)), graph=args.graph)
    e2e_gbs = world * sum(e2e_bytes) / (sum(e2e_ms) * 1e-3) / 1e9
    zc_ms, zc_bytes, zc_h2d, zc_d2h = time_e2e_zero_copy(cfg, items, max(5, min(args.steps, 20)))
    zc_gbs = world * sum(zc_bytes) / (sum(zc_ms) * 1e-3) / 1e9

    per_config = {}
    if world == 1 and not args.no_extra:
        for name in args.extra.split(","):
            if not name or name == args.config:
                continue
            c = CONFIGS[name]
            it2 = workload(c)
            m2, b2 = time_layer(c, it2, max(10, min(args.steps, 40)), 3, graph=args.graph)
            g2 = sum(b2) / (sum(m2) * 1e-3) / 1e9
            per_config[name] = {"ms_per_step": round(statistics.mean(m2), 5), "weight_gbs": round(g2, 1),
                                "roof_frac": round(g2 / peak, 4),
                                "mean_active_experts": statistics.mean(i["G"] for i in it2),
                                "rows": statistics.mean(i["R"] for i in it2)}
    # the GEMV path (W4A16, exact bf16 activations): a validation path, timed on the same workload
    w4a16 = None
    if world == 1 and not args.no_extra:
        m3, b3 = time_w4a16(cfg, items, max(10, min(args.steps, 40)))
        g3 = sum(b3) / (sum(m3) * 1e-3) / 1e9
        w4a16 = {"workload": cfg.name, "ms_per_step": round(statistics.mean(m3), 5), "weight_gbs": round(g3, 1),
                 "roof_frac": round(g3 / peak, 4), "launches_per_step": 5}
    # route, gather+quantize (one launch when T*k <= 32), the w13+w2 grouped GEMM (one
    # persistent launch), scatter
    launches_per_step = 3 if max(i["T"] for i in items) * cfg.k <= 32 else 4
    out = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "ms_per_step_median": round(statistics.median(ms), 5),
        "step_launch": ("CUDA graph of the C-ABI call (one per routing buffer set)" if args.graph else
                        "direct C-ABI call (its kernels chained by programmatic dependent launch)"),
        ("ms_per_step_direct" if args.graph else "ms_per_step_graph"): round(statistics.mean(ms_other), 5),
        "ms_per_step_code_warm": round(statistics.mean(ms_warm), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate)",
        "data": "synthetic (seeded; NVFP4 codes drawn directly, bf16 activations N(0,1))",
        "config": {
            "workload": f"{cfg.name}: {cfg.E} experts, hidden {cfg.H}, intermediate {cfg.I}, "
                        + (f"{cfg.T} token(s) top-{cfg.k}" if cfg.routing == "topk" else
                           f"all experts, Mg~U{{{cfg.mg_lo}..{cfg.mg_hi}}}"),
            "mean_active_experts": statistics.mean(i["G"] for i in items),
            "rows_per_step": statistics.mean(i["R"] for i in items),
            "bytes_per_step": statistics.mean(byts),
            "l2": "flushed before every timed step (write of a 2x-L2 buffer, then a read of another); "
                  "routing rotated over 20 seeded draws",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roof_frac": round(gbs / world / peak, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": "gemm_kernel (w13 + SwiGLU/requantize, then w2: one launch)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(),
            "algorithmic_bytes_per_launch": round(gemm_bytes),
        },
        "stage_ms": {k: round(v, 5) for k, v in stages.items()},
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "ms_per_step": round(statistics.mean(e2e_ms), 5),
                "h2d_bytes_per_step": round(h2d), "d2h_bytes_per_step": round(d2h)},
        "e2e_host_buffers_in_place": {
            "value": round(zc_gbs, 2), "unit": "GB/s", "ms_per_step": round(statistics.mean(zc_ms), 5),
            "h2d_bytes_per_step": round(zc_h2d), "d2h_bytes_per_step": round(zc_d2h),
            "how": "x, routing, router weights and y in pinned host memory passed to the call as they are "
                   "(unified addressing): the kernels read and write them over the CPU-GPU link, no copy queued"},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "per_config": per_config,
        "w4a16_gemv_path": w4a16,
        "device": props.name,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.config)
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (the reported baseline, and the reference arm)
# ---------------------------------------------------------------------------

def oracle_tasks(cfg_name, step_index):
    """The oracle's work for one layer step of the config's first token: one
    task per routed slot (the token's experts; for decode M=1 that is the
    whole top-8 step). Returns (task list, algorithmic bytes of the step)."""
    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_routing

    cfg = CONFIGS[cfg_name]
    ids, _ = make_routing(cfg, seed=2 + 1000 * step_index)
    slots = [j for j in range(ids.shape[1]) if 0 <= int(ids[0, j]) < cfg.E]
    return [(step_index, j) for j in slots], step_bytes(cfg, len(slots), 1)


def oracle_worker(cfg_name, worker, warm, timed, ready, go, done, out):
    """One spawned process, one thread: prepares its tasks' inputs (one
    synthetic expert's NVFP4 weights, seeded by the worker, reused by every
    task, and each task's token row and router weight), then, between the
    parent's barriers, runs the oracle's layer step of every task: that
    token routed to that one expert."""
    import numpy as np
    import torch

    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_activations, make_routing, make_weights
    from oracle import nvfp4_moe as O

    cfg = CONFIGS[cfg_name]
    w = {k: v.numpy() for k, v in make_weights(1, cfg.H, cfg.I, seed=3 + worker).items()}

    def prepare(task):
        step, j = task
        ids, tw = make_routing(cfg, seed=2 + 1000 * step)
        one = np.full((1, cfg.k), -1, np.int32)
        one[0, j] = 0                                   # the slot's expert, renumbered 0
        x = make_activations(1, cfg.H, seed=1 + 1000 * step).view(torch.int16).numpy().view(np.uint16)
        return x, one, tw[:1].numpy()

    warm_in = [prepare(t) for t in warm]
    timed_in = [prepare(t) for t in timed]
    for x, ids, tw in warm_in:
        O.moe_layer(x, ids, tw, w, E=1)
    ready.wait()
    go.wait()                                           # the timed region starts for every worker at once
    for x, ids, tw in timed_in:
        O.moe_layer(x, ids, tw, w, E=1)
    done.wait()
    out.put(worker)


def oracle_parallel(cfg_name, workers, steps, warmup):
    """Times `steps` oracle layer steps (after `warmup`) of the config's first
    token, every routed expert a task, tasks dealt round-robin over `workers`
    spawned single-thread processes. Inputs are prepared before the timed
    region; the wall clock runs from a barrier all workers wait at to the
    last task done. Returns (bytes, seconds, description)."""
    import multiprocessing as mp

    warm_tasks, timed_tasks, total_bytes = [], [], 0
    for i in range(warmup):
        warm_tasks += oracle_tasks(cfg_name, i)[0]
    for i in range(warmup, warmup + steps):
        t, b = oracle_tasks(cfg_name, i)
        timed_tasks += t
        total_bytes += b
    ctx = mp.get_context("spawn")
    ready, go, done = ctx.Barrier(workers + 1), ctx.Barrier(workers + 1), ctx.Barrier(workers + 1)
    out = ctx.Queue()
    env_keep = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in env_keep:
        os.environ[v] = "1"                             # one thread per worker (inherited at spawn)
    procs = [ctx.Process(target=oracle_worker,
                         args=(cfg_name, r, warm_tasks[r::workers], timed_tasks[r::workers], ready, go, done, out))
             for r in range(workers)]
    try:
        for p in procs:
            p.start()
        ready.wait()
        go.wait()
        t0 = time.perf_counter()
        done.wait()
        sec = time.perf_counter() - t0
        for p in procs:
            p.join()
    finally:
        for v, val in env_keep.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val
    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS
    cfg = CONFIGS[cfg_name]
    per = len(timed_tasks) // max(1, steps)
    desc = (f"{steps} step(s) of {cfg_name}'s first token (top-{cfg.k}: {per} expert tasks per step, hidden "
            f"{cfg.H}, intermediate {cfg.I}), each task the oracle's layer step for one routed expert, "
            f"{workers} spawned single-thread process(es), tasks dealt round-robin")
    return total_bytes, sec, desc


def oracle_child(args):
    """Runs in a fresh process (no CUDA context): the parallel oracle timing."""
    b, s, desc = oracle_parallel(args.config, args.child_workers, args.child_steps, args.child_warmup)
    print(json.dumps({"bytes": b, "seconds": s, "steps": args.child_steps, "workers": args.child_workers,
                      "desc": desc}))


def run_oracle_child(config, workers, steps, warmup):
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", "--config", config,
           "--child-workers", str(workers), "--child-steps", str(steps), "--child-warmup", str(warmup)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(config):
    """The oracle on the host cores: all of them (one process per core, the
    reported figure) and one (single_core), each over whole steps of the
    config's first token (for decode M=1: the full top-8 step)."""
    n = host_cores()
    res = run_oracle_child(config, n, steps=max(2, (2 * n) // 8 * 2), warmup=1)
    one = run_oracle_child(config, 1, steps=2, warmup=1)
    entry = lambda r: {"value": round(r["bytes"] / r["seconds"] / 1e9, 4), "unit": "GB/s",  # noqa: E731
                       "cores": r["workers"], "kind": "oracle", "sample": r["desc"],
                       "ms_per_step": round(1e3 * r["seconds"] / r["steps"], 1)}
    out = entry(res)
    out["cpu_model"] = cpu_model()
    out["single_core"] = entry(one)
    return out


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def reference_arm(args, rank, world):
    """The CPU oracle as the reference arm: the same metric on whole steps of
    the config's first token (for decode M=1 the full top-8 step), on every
    host core (one spawned process per core). Rank 0 only."""
    if rank != 0:
        return
    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS
    cfg = CONFIGS[args.config]
    n = host_cores()
    res = run_oracle_child(args.config, n, steps=args.steps, warmup=args.warmup)
    gbs = res["bytes"] / res["seconds"] / 1e9
    ms = 1e3 * res["seconds"] / res["steps"]
    sample = f"{res['steps']} timed step(s) after {args.warmup} warm-up: {res['desc']}"
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle; fp32 codec divisions)",
        "data": "synthetic",
        "config": {"workload": f"{cfg.name}: {cfg.E} experts, hidden {cfg.H}, intermediate {cfg.I}",
                   "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": res["workers"], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode_m1")
    ap.add_argument("--extra", default="decode_m8,decode_m32,full_stream,large_batch,prefill_m32",
                    help="further configs timed on one GPU and reported under per_config")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--profile", action="store_true", help="short run for ncu: warm-up and timed steps only")
    ap.add_argument("--path", default="w4a4", choices=["w4a4", "w4a16"],
                    help="with --profile: the grouped path (w4a4) or the GEMV path (w4a16)")
    ap.add_argument("--graph", action="store_true", help="time CUDA-graph replays of the call instead of direct calls")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (small profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--child-workers", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--child-steps", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--child-warmup", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup) if not args.oracle_child else args.warmup
    if args.oracle_child:
        oracle_child(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_bench(args, rank, world)


if __name__ == "__main__":
    main()
