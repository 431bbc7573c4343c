#!/usr/bin/env python3
"""Throughput of the routed MoE layer forward on B300, against the roofline and the CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole hot path over one batch of synthetic input,
through the library's layer call (ftmoe_layer_forward):
  * route (logits, top-k, weights);
  * permute (expert-sorted pairs);
  * the expert FFN;
  * the weighted combine to bf16;
plus the global-LRU access of the step's experts (ftmoe_slot_lru) on a side
stream.  The FFN is timed with the step's experts resident.  In the `stack`
workloads a step runs the batch through all 8 layers.

Default workload: decode, 128 experts top-8, d 2048, ffn 768, NVFP4, batch 1
(MoE-layer tokens/s at decode).  Successive steps cycle through 16 distinct
layer weight sets (5.4 GB).  A layer's weights are re-read only after 15
other layers' worth of traffic, so its bytes come from HBM, not from the
126 MB L2.

Output: one JSON line (rank 0).  Under torchrun every rank runs its own
replica on its own GPU ("scaling": "weak").  The value is the sum over ranks
of tokens / (max over ranks of the timed region).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOADS = {
    # name: (Workload, tokens per step, layer copies cycled)
    "decode": (synth.DECODE, 1, 16),
    "decode4": (synth.DECODE, 4, 16),
    "decode16": (synth.DECODE, 16, 16),
    "prefill": (synth.PREFILL, 8192, 2),
    "stack1": (synth.STACK, 1, 8),
    "stack16": (synth.STACK, 16, 8),
    "stack64": (synth.STACK, 64, 8),
    "prefill_split": (synth.PREFILL_SPLIT, 16384, 1),
    "tiny": (synth.TINY, 16, 64),
}
METRIC = "MoE-layer tokens/s"
DEFAULT_STEPS = {"decode": 40000, "decode4": 30000, "decode16": 20000, "prefill": 1000, "stack1": 4000,
                 "stack16": 2000, "stack64": 1000, "prefill_split": 200, "tiny": 40000}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: per workload, about a second)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="layer copies to cycle (decode workloads; default 16)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU baseline sample")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (a smaller case of the same kernels, for profiler captures)")
    ap.add_argument("--no-cache-legs", action="store_true",
                    help="skip the expert-cache (fills, q* split) and streamed-prefill reports")
    ap.add_argument("--prefill-steps", type=int, default=200,
                    help="timed steps of the 8192-token prefill leg that the default decode run reports beside "
                         "its headline (0 = skip the leg)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: independent replicas, no data-path collective)
# ---------------------------------------------------------------------------
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------
class Layer:
    def __init__(self, wl: synth.Workload, seed: int, device):
        L = wl.layer
        self.W = synth.make_experts(L.fmt, L.E, L.d, L.f, seed, device=device)
        self.wr = synth.make_router(L.E, L.d, seed, device=device)
        self.bias = torch.from_numpy(synth.make_zipf_bias(L.E, wl.zipf_s, seed)).to(device)


def expert_bytes(wl):
    return synth.expert_bytes(wl.layer.fmt, wl.layer.d, wl.layer.f)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def kernel_hash() -> str:
    d = os.path.join(ROOT, "sparse_moe_expert_sorted_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per FFN call from the committed ncu summary, if it was taken on the current kernels."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(workload)
    if not ent or ent.get("kernel_hash") != kernel_hash():
        return None
    return ent.get("bytes_per_call")


def new_graph():
    try:
        return torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        return torch.cuda.CUDAGraph()


def graph_kernel_nodes(graph):
    """Kernel nodes of a captured graph (every one is a launch of this library), or None."""
    try:
        from cuda.bindings import runtime as rt
        g = graph.raw_cuda_graph()
        err, _, n = rt.cudaGraphGetNodes(g, 0)
        if int(err) != 0:
            return None
        err, nodes, n = rt.cudaGraphGetNodes(g, n)
        if int(err) != 0:
            return None
        kern = 0
        for nd in nodes:
            err, typ = rt.cudaGraphNodeGetType(nd)
            if int(err) == 0 and int(typ) == int(rt.cudaGraphNodeType.cudaGraphNodeTypeKernel):
                kern += 1
        return kern
    except Exception:
        return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def bench_ours(args, rank, ws):
    import sparse_moe_expert_sorted_b300 as ft
    ft.lib()  # fails loudly if the library is missing
    wl, T, n_layers = WORKLOADS[args.workload]
    if args.layers and not args.workload.startswith("stack"):
        n_layers = args.layers
    if args.experts:
        import dataclasses
        wl = dataclasses.replace(wl, layer=dataclasses.replace(wl.layer, E=args.experts),
                                 capacity=min(wl.capacity, args.experts) if wl.capacity else 0)
    L = wl.layer
    dev = "cuda"
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
    stack = args.workload.startswith("stack")
    layers = [Layer(wl, 1000 * (rank + 1) + i, dev) for i in range(n_layers)]
    n_x = 64
    xs = [synth.make_x(T, L.d, 77 + 1000 * rank + i, device=dev) for i in range(n_x)]
    P = T * L.k
    nl_step = n_layers if stack else 1
    # ids / weights per (buffer b, layer in the step): the side stream's LRU reads step i's ids
    # while step i + 1 runs, so steps alternate between two buffers
    ids = [[torch.empty(T, L.k, dtype=torch.int32, device=dev) for _ in range(nl_step)] for _ in range(2)]
    tw = [[torch.empty(T, L.k, dtype=torch.float32, device=dev) for _ in range(nl_step)] for _ in range(2)]
    off = torch.empty(L.E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(P, dtype=torch.int32, device=dev)
    y = torch.empty(P, L.d, dtype=torch.float32, device=dev)
    out = torch.empty(T, L.d, dtype=torch.float32, device=dev)
    out_bf = torch.empty(T, L.d, dtype=torch.bfloat16, device=dev)
    ws_r = ft.workspace(ft.route_workspace_size(dsc, T))
    ws_p = ft.workspace(ft.permute_workspace_size(dsc, T))
    ws_f = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    ws_l = ft.workspace(ft.layer_workspace_size(dsc, T))
    path = ft.expert_ffn_path(dsc, T)
    for l in layers:   # derived layouts the fast kernels read (prepared once, outside timing)
        ft.prepare_weights(dsc, l.W)
    structs = [ft.weights_struct(l.W) for l in layers]
    lru = ft.LRU(wl.layers if stack else 1, L.E, wl.capacity or L.E)
    cap = min(P, L.E)
    hit = torch.empty(cap, dtype=torch.uint8, device=dev)
    lslot = torch.empty(cap, dtype=torch.int32, device=dev)
    lev = torch.empty(cap, dtype=torch.int32, device=dev)
    lcnt = torch.zeros(2, dtype=torch.int64, device=dev)
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    ev_main = [[torch.cuda.Event() for _ in range(nl_step)] for _ in range(2)]
    ev_side = [[torch.cuda.Event() for _ in range(nl_step)] for _ in range(2)]

    recorded = set()     # (b, j) whose side event was recorded in the current capture / warm-up

    def one_layer(li, x, j, b):
        """Layer li through ftmoe_layer_forward (route, permute, expert FFN, combine) on the main
        stream; the global-LRU access of its experts on the side stream."""
        l = layers[li]
        if (b, j) in recorded:
            main.wait_event(ev_side[b][j])   # the LRU of two steps ago has read ids[b][j]
        ft.layer_forward(dsc, structs[li], None, x, l.wr, l.bias, ids[b][j], tw[b][j], out, out_bf, ws_l, main)
        ev_main[b][j].record(main)
        side.wait_event(ev_main[b][j])
        lru.step(j if stack else 0, ids[b][j], hit, lslot, lev, lcnt, side)
        ev_side[b][j].record(side)
        recorded.add((b, j))

    def step(i):
        x = xs[i % n_x]
        b = i % 2
        if stack:
            for li in range(n_layers):
                one_layer(li, x, li, b)
        else:
            one_layer(i % n_layers, x, 0, b)

    def join_side():
        for b, j in sorted(recorded):
            main.wait_event(ev_side[b][j])
        recorded.clear()

    # eager warm-up (also loads every kernel), then capture K steps into one graph
    with torch.cuda.stream(main):
        for i in range(max(1, args.warmup)):
            step(i)
        join_side()
    torch.cuda.synchronize()

    K = args.steps
    # one graph of G steps, replayed K / G times inside the timed region (G divides K)
    G = min(K, 1000)
    while K % G:
        G -= 1
    graph = new_graph()
    with torch.cuda.graph(graph, stream=main):
        for i in range(G):
            step(i)
        join_side()
    nodes = graph_kernel_nodes(graph)
    launches_in_graph = None if nodes is None else nodes * (K // G)
    with torch.cuda.stream(main):     # replay() launches on the current stream
        for _ in range(max(3, args.warmup // max(1, G) + 1)):
            graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(main):
        t0.record(main)
        for _ in range(K // G):
            graph.replay()
        t1.record(main)
    t1.synchronize()
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, ws)
    tokens = T * K * ws
    value = tokens / (ms_max / 1e3)
    gpu_launches = launches_in_graph

    lpath = ft.layer_path(dsc, structs[0], T)
    fused = lpath in (1, 2)
    peaks, src = load_peaks()
    hbm = peaks["hbm_gbs"]
    eb = expert_bytes(wl)
    if fused:
        # --- the step's one kernel (router + expert FFN + merge) timed per launch ---
        layer_us, uniq_l = time_layer_calls(ft, dsc, layers, structs, xs, T, L, n_layers, min(G, 256), ws_l, main)
        alg_bytes = uniq_l * eb + L.E * L.d * 2 + T * L.d * 2 + T * L.d * (4 + 2)
        achieved = alg_bytes / (layer_us / 1e6) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "traffic": ncu_traffic(args.workload),
                    "kernel": "ftmoe_layer_forward (one launch: " + ("sl_layer_kernel, the one-token slice form"
                                                                   if lpath == 2 else
                                                                   "sd_ffn_kernel with the router fused") + ")",
                    "peak_source": src, "kernel_us": round(layer_us, 3), "alg_bytes_per_call": int(alg_bytes),
                    "mean_unique_experts": round(uniq_l, 2)}
        e2e = bench_e2e(ft, dsc, layers, structs, T, L, wl, stack, n_layers, e2e_steps(K, T), main)
        return finish(args, ws, wl, L, T, K, ms_max, value, stack, n_layers, eb, roofline, e2e, gpu_launches, clk,
                      lru)

    # --- dominant call (expert FFN) timed alone over the same steps ----------
    n_ffn = min(G, 256)
    sev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_ffn)]
    eev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_ffn)]
    uniq = []
    g2 = torch.cuda.CUDAGraph()
    routes = []
    with torch.cuda.stream(main):
        for i in range(n_ffn):
            li = i % n_layers
            x = xs[i % n_x]
            l = layers[li]
            r_ids = torch.empty(T, L.k, dtype=torch.int32, device=dev)
            r_w = torch.empty(T, L.k, dtype=torch.float32, device=dev)
            r_off = torch.empty_like(off)
            r_sp = torch.empty_like(sp)
            r_pp = torch.empty_like(sp)
            ft.route(dsc, x, l.wr, l.bias, r_ids, r_w, None, ws_r, main)
            ft.permute(dsc, r_ids, r_off, r_sp, r_pp, ws_p, main)
            routes.append((li, x, r_ids, r_off, r_sp, r_w))
    torch.cuda.synchronize()
    for li, x, r_ids, r_off, r_sp, r_w in routes:
        uniq.append(len(np.unique(r_ids.cpu().numpy())))
    out.zero_()
    with torch.cuda.graph(g2, stream=main):
        for i, (li, x, r_ids, r_off, r_sp, r_w) in enumerate(routes):
            sev[i].record(main)
            ft.expert_ffn(dsc, structs[li], None, x, r_off, r_sp, r_w, out, ws_f, main)
            eev[i].record(main)
    with torch.cuda.stream(main):
        g2.replay()
        g2.replay()
    torch.cuda.synchronize()
    ffn_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(sev, eev)]))
    alg_bytes = float(np.mean(uniq)) * eb + T * L.d * 2 + P * L.d * 4
    achieved = alg_bytes / (ffn_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": ncu_traffic(args.workload),
                "kernel": "ftmoe_expert_ffn (decode: sd_ffn_kernel, one launch)", "peak_source": src,
                "ffn_us": round(ffn_ms * 1e3, 3), "alg_bytes_per_call": int(alg_bytes),
                "mean_unique_experts": round(float(np.mean(uniq)), 2)}
    if path != 0:
        flops = 2.0 * P * 3 * L.d * L.f
        ratio = 6.0 if path == 1 else 2.0   # nominal FP4:bf16 and FP8:bf16 dense ratios
        peak_t = peaks["bf16_tflops"] * ratio
        ach = flops / (ffn_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": round(peak_t, 1), "unit": "TFLOP/s",
                    "frac": round(ach / peak_t, 4), "traffic": ncu_traffic(args.workload),
                    "kernel": "ftmoe_expert_ffn (quantise, gather, gate/up GEMM, down GEMM)",
                    "peak_source": f"{src} bf16 x {ratio:g} (nominal ratio)",
                    "ffn_us": round(ffn_ms * 1e3, 3)}

    # --- end to end through the public API with host buffers ------------------
    e2e = bench_e2e(ft, dsc, layers, structs, T, L, wl, stack, n_layers, e2e_steps(K, T), main)
    return finish(args, ws, wl, L, T, K, ms_max, value, stack, n_layers, eb, roofline, e2e, gpu_launches, clk, lru)


def time_layer_calls(ft, dsc, layers, structs, xs, T, L, n_layers, n, ws_l, main):
    """Mean device time of one ftmoe_layer_forward launch: a captured sequence of n launches
    that cycles the layer copies, timed by CUDA events before its first and after its last
    launch on their stream (events between launches would hold each launch back until the
    previous one has finished, hiding nothing of its launch latency), divided by n; and the
    mean count of distinct experts."""
    dev = "cuda"
    ev0 = torch.cuda.Event(enable_timing=True, external=True)
    ev1 = torch.cuda.Event(enable_timing=True, external=True)
    ids = [torch.empty(T, L.k, dtype=torch.int32, device=dev) for _ in range(n)]
    tw = torch.empty(T, L.k, dtype=torch.float32, device=dev)
    out = torch.empty(T, L.d, dtype=torch.float32, device=dev)
    out_bf = torch.empty(T, L.d, dtype=torch.bfloat16, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        ev0.record(main)
        for i in range(n):
            l = layers[i % n_layers]
            ft.layer_forward(dsc, structs[i % n_layers], None, xs[i % len(xs)], l.wr, l.bias, ids[i], tw, out, out_bf,
                             ws_l, main)
        ev1.record(main)
    with torch.cuda.stream(main):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    us = ev0.elapsed_time(ev1) * 1e3 / n
    uniq = float(np.mean([len(np.unique(t.cpu().numpy())) for t in ids]))
    return us, uniq


def finish(args, ws, wl, L, T, K, ms_max, value, stack, n_layers, eb, roofline, e2e, gpu_launches, clk, lru):
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_max / K, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {0: "bf16", 1: "nvfp4", 2: "mxfp4", 3: "fp8_e4m3"}[L.fmt] + " weights, fp32 accumulate",
        "data": "synthetic (seeded; random-init weights)",
        "config": {"workload": f"{wl.name} T={T}" + (" x8 layers" if stack else "") +
                               (f" (E overridden to {L.E})" if args.experts else ""), "E": L.E, "k": L.k,
                   "d": L.d, "ffn": L.f, "tokens_per_step": T, "layers_cycled": n_layers,
                   "l2": f"weights > L2: {n_layers} distinct layer copies cycled "
                         f"({n_layers * L.E * eb / 1e9:.1f} GB)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roofline, "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clk,
    }
    lru.close()
    if not args.experts:
        try:
            res["lru_replay"] = lru_replay(wl, T, stack)
        except Exception as e:     # the replay is a side report: never lose the bench line over it
            res["lru_replay"] = {"error": str(e)[:200]}
    return res


def lru_replay(wl, T, stack, dev="cuda"):
    """The workload's routing trace (Gumbel-top-k over the Zipf ranks) replayed through the
    global LRU in one ftmoe_slot_lru_replay launch from a cold table: access and miss counts,
    and the device time of the replay (CUDA events, best of 3 cold-start replays)."""
    import sparse_moe_expert_sorted_b300 as ft
    if not wl.capacity or not wl.trace_steps:
        return None
    L = wl.layer
    nl = wl.layers if stack else 1
    trace = synth.make_trace(wl.trace_steps, nl, T, L.k, L.E, wl.zipf_s, seed=wl.seed)
    steps = trace.shape[0]
    cap = steps * nl * min(T * L.k, L.E)
    h = ft.LRU(nl, L.E, wl.capacity)
    try:
        tr = torch.from_numpy(np.ascontiguousarray(trace)).to(dev)
        hit = torch.empty(cap, dtype=torch.uint8, device=dev)
        slot = torch.empty(cap, dtype=torch.int32, device=dev)
        ev = torch.empty(cap, dtype=torch.int32, device=dev)
        cnt = torch.zeros(2, dtype=torch.int64, device=dev)
        h.replay(tr, hit, slot, ev, cnt)
        acc, miss = (int(v) for v in cnt.tolist())
        times = []
        for _ in range(3):
            h.reset()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            h.replay(tr, hit, slot, ev, cnt)
            t1.record()
            t1.synchronize()
            times.append(t0.elapsed_time(t1))
        again = [int(v) for v in cnt.tolist()]
    finally:
        h.close()
    return {"trace_steps": steps, "layers": nl, "tokens_per_step": T, "experts_per_token": L.k,
            "capacity": wl.capacity, "accesses": acc, "misses": miss, "miss_rate": round(miss / max(1, acc), 4),
            "repeatable": again == [acc, miss], "replay_us_per_step": round(min(times) * 1e3 / steps, 3),
            "how": "one ftmoe_slot_lru_replay launch per replay, cold start; synthetic iid Zipf trace"}


def e2e_steps(K, T):
    """Steps of the end-to-end leg: enough for ~50 ms of one-token steps, 200 of the long ones."""
    return min(K, 2000 if T <= 64 else 200)


def bench_e2e(ft, dsc, layers, structs, T, L, wl, stack, n_layers, steps, main):
    """Same metric through the public API with pinned host inputs and outputs.  Per step the
    host-buffer layer call: H2D of x, the layer, D2H of the bf16 output.  The one-call
    workloads replay it as a CUDA graph recorded once per buffer set (ftmoe_layer_graph_*) and
    also time the direct call (ftmoe_layer_forward_host, one prepared ctypes call per step);
    the stack workloads copy x once and run the 8 layers on it.  Wall clock over the steps, and
    the host time spent issuing them."""
    dev = "cuda"
    xh = [synth.make_x(T, L.d, 555 + i).pin_memory() for i in range(8)]
    oh = torch.empty(T, L.d, dtype=torch.bfloat16).pin_memory()
    of = torch.empty(T, L.d, dtype=torch.float32, device=dev)
    ob = torch.empty(T, L.d, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(T, L.k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, L.k, dtype=torch.float32, device=dev)

    def run(step):
        for i in range(5):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            step(i)
        t_issue = time.perf_counter() - t0
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        return round(T * steps / dt, 3), round(t_issue * 1e6 / steps, 2)

    extra = {}
    if stack:
        xd = torch.empty(T, L.d, dtype=torch.bfloat16, device=dev)
        ws = ft.workspace(ft.layer_workspace_size(dsc, T))

        def step(i):
            with torch.cuda.stream(main):
                xd.copy_(xh[i % len(xh)], non_blocking=True)
                for li in range(n_layers):
                    l = layers[li]
                    ft.layer_forward(dsc, structs[li], None, xd, l.wr, l.bias, ids, tw, of, ob, ws, main)
                oh.copy_(ob, non_blocking=True)
        how = "per step: pinned H2D of x, ftmoe_layer_forward per layer, D2H of the bf16 output; wall clock"
        value, issue = run(step)
    else:
        # two streams, each with its own workspace and output buffers, take alternate steps, as a
        # serving loop would: one step's host copies overlap the other's compute (the link is
        # full duplex).  Every step still copies its own x in and its own output out.
        streams = [main, torch.cuda.Stream()]
        wss = [ft.workspace(ft.layer_host_workspace_size(dsc, T)) for _ in streams]
        ohs = [oh, torch.empty(T, L.d, dtype=torch.bfloat16).pin_memory()]
        dev_out = [(ids, tw, of), (torch.empty_like(ids), torch.empty_like(tw), torch.empty_like(of))]
        key = lambda i: (i % len(xh), i % n_layers, i % 2)
        keys = sorted({key(i) for i in range(steps + 5)})
        calls, graphs, graph_error = {}, {}, None
        for k_ in keys:
            i, li, j = k_
            l = layers[li]
            i_, w_, o_ = dev_out[j]
            a_ = (dsc, structs[li], None, xh[i], l.wr, l.bias, i_, w_, o_, ohs[j], wss[j])
            calls[k_] = ft.LayerHostCall(*a_, streams[j])
            if graph_error is None:
                try:
                    graphs[k_] = ft.LayerHostGraph(*a_, stream=streams[j])
                except ft.FtmoeError as e:   # reported in the line; the direct calls still measure e2e
                    graph_error = str(e)
        d_value, d_issue = run(lambda i: calls[key(i)]())
        direct_how = ("per step: one ftmoe_layer_forward_host call (pinned H2D of x, the layer, D2H of the bf16 "
                      "output), arguments packed once; steps alternate between two streams with their own "
                      "buffers; wall clock")
        if graph_error is None:
            value, issue = run(lambda i: graphs[key(i)]())
            how = ("per step: one replay of a CUDA graph that holds one ftmoe_layer_forward_host call (pinned H2D "
                   "of x, the layer, D2H of the bf16 output), recorded once per buffer set by "
                   "ftmoe_layer_graph_create; steps alternate between two streams with their own buffers; wall clock")
            extra = {"direct_calls": {"value": d_value, "host_issue_us_per_step": d_issue, "how": direct_how}}
        else:
            value, issue, how = d_value, d_issue, direct_how
            extra = {"graph_error": graph_error}
        for g in graphs.values():
            g.close()
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": T * L.d * 2,
            "d2h_bytes_per_step": T * L.d * 2, "steps": steps, "host_issue_us_per_step": issue, "how": how, **extra}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_rate(workload: str, budget_s: float, max_steps: int | None = None):
    """Oracle tokens/s on a bounded sample of the workload (host cores)."""
    from oracle import ffn as OF
    wl, T, n_layers = WORKLOADS[workload]
    L = wl.layer
    stack = workload.startswith("stack")
    # one layer's weights on the host; the oracle dequantises each expert inside the timed region
    Wt = synth.make_experts(L.fmt, L.E, L.d, L.f, 4242, device="cuda" if torch.cuda.is_available() else "cpu")
    W = dict(fmt=L.fmt, d=L.d, f=L.f, glob=Wt.glob.cpu().numpy())
    for name in ("gate", "up", "down"):
        t = getattr(Wt, name).cpu()
        W[name] = t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
        s = getattr(Wt, name + "_s")
        W[name + "_s"] = None if s is None else s.cpu().numpy()
    del Wt
    wr = synth.make_router(L.E, L.d, 4242).view(torch.int16).numpy().view(np.uint16)
    bias = synth.make_zipf_bias(L.E, wl.zipf_s, 4242)
    slot = np.arange(L.E)
    sample_T = T if T <= 64 else 256                       # prefill: a 256-token sample of the chunk
    done_tokens = 0
    steps = 0
    t0 = time.perf_counter()
    while True:
        x = synth.make_x(sample_T, L.d, 900 + steps).view(torch.int16).numpy().view(np.uint16)
        for _ in range(n_layers if stack else 1):
            OF.layer(W, slot, x, wr, bias, L.k, L.renorm)
        done_tokens += sample_T
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and steps >= max_steps):
            break
    threads = blas_threads()
    sample = (f"{steps} oracle step(s) of {sample_T} token(s)" + (" x 8 layers" if stack else "") +
              f" ({'the full batch' if sample_T == T else f'a {sample_T}-token sample of the {T}-token chunk'})")
    return done_tokens / el, threads, sample, el


def blas_threads() -> int:
    """Threads numpy's BLAS uses (the oracle's matmuls); else the usable cores."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def bench_reference(args, rank, ws):
    wl, T, n_layers = WORKLOADS[args.workload]
    budget = 20.0     # seconds of oracle work: a bounded sample of the workload
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_rate(args.workload, 0.0, max_steps=1)
    rate, threads, sample, el = oracle_rate(args.workload, budget, max_steps=args.steps)
    value = rate
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * T / rate, 3) if rate else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": f"{wl.name} T={T}" + (" x8 layers" if args.workload.startswith("stack") else ""),
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def link_and_host_bandwidth(dev="cuda"):
    """The two bandwidths of the q* policy, measured on this machine: B_P, the host link
    (pinned host -> device copies, 256 MiB, best of 3), and B_H, the host memory (a 1 GiB
    copy between host buffers by as many threads as the process may use)."""
    import concurrent.futures as cf
    n = 256 << 20
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        e1.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, d
    m = 1 << 30
    a = np.ones(m, np.uint8)
    b = np.empty_like(a)
    nt = max(1, len(os.sched_getaffinity(0)))
    parts = np.array_split(np.arange(m), nt)
    bounds = [(int(p[0]), int(p[-1]) + 1) for p in parts if len(p)]

    def cp(lo_hi):
        lo, hi = lo_hi
        np.copyto(b[lo:hi], a[lo:hi])

    host = 0.0
    with cf.ThreadPoolExecutor(nt) as ex:
        list(ex.map(cp, bounds))
        for _ in range(3):
            t0 = time.perf_counter()
            list(ex.map(cp, bounds))
            host = max(host, 2 * m / (time.perf_counter() - t0) / 1e9)   # read + write bytes
    return round(best, 2), round(host, 2), nt


def cache_leg(steps=300, dev="cuda"):
    """Decode steps with the 37% slot table: the expert pool in pinned host memory, the LRU's
    misses filled into HBM slots, and the q* split between executor A (HBM slots) and
    executor B (streaming the other experts from the host pool), merged exactly.  Tokens/s per
    policy (q* from the measured bandwidths, fill every miss, fill none), miss counts, and the
    fill kernel's bandwidth against the host link."""
    import sparse_moe_expert_sorted_b300 as ft
    wl = synth.DECODE
    L = wl.layer
    T, C = 1, wl.capacity
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
    Wp = synth.make_experts(L.fmt, L.E, L.d, L.f, 4321, device=dev)
    pin = lambda t: None if t is None else t.cpu().contiguous().pin_memory()
    pool = synth.ExpertWeights(Wp.fmt, Wp.d, Wp.f, pin(Wp.gate), pin(Wp.up), pin(Wp.down), pin(Wp.gate_s),
                               pin(Wp.up_s), pin(Wp.down_s), pin(Wp.glob))
    del Wp
    ft.prepare_weights(dsc, pool)
    z = lambda t: None if t is None else torch.zeros((C,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
    arena = synth.ExpertWeights(pool.fmt, pool.d, pool.f, z(pool.gate), z(pool.up), z(pool.down), z(pool.gate_s),
                                z(pool.up_s), z(pool.down_s), z(pool.glob))
    ft.prepare_weights(dsc, arena)
    s_fill, s_pool, s_arena = ft.weights_struct(pool), ft.weights_struct(pool, prepared=0), ft.weights_struct(arena)
    wr = synth.make_router(L.E, L.d, 4321, device=dev)
    bias = torch.from_numpy(synth.make_zipf_bias(L.E, wl.zipf_s, 4321)).to(dev)
    xs = [synth.make_x(T, L.d, 8000 + i, device=dev) for i in range(64)]
    P, n = T * L.k, min(T * L.k, L.E)
    ids = torch.empty(T, L.k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, L.k, dtype=torch.float32, device=dev)
    off = torch.empty(L.E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(P, dtype=torch.int32, device=dev)
    pp = torch.empty(P, dtype=torch.int32, device=dev)
    hit = torch.empty(n, dtype=torch.uint8, device=dev)
    lslot = torch.empty(n, dtype=torch.int32, device=dev)
    lev = torch.empty(n, dtype=torch.int32, device=dev)
    sa = torch.empty(L.E, dtype=torch.int32, device=dev)
    sb = torch.empty(L.E, dtype=torch.int32, device=dev)
    now = torch.empty(n, 2, dtype=torch.int32, device=dev)
    later = torch.empty(n, 2, dtype=torch.int32, device=dev)
    cnt = torch.zeros(4, dtype=torch.int32, device=dev)
    tot = torch.zeros(4, dtype=torch.int64, device=dev)
    y_a = torch.empty(P, L.d, dtype=torch.float32, device=dev)
    out_b = torch.empty(T, L.d, dtype=torch.float32, device=dev)
    of = torch.empty(T, L.d, dtype=torch.float32, device=dev)
    ob = torch.empty(T, L.d, dtype=torch.bfloat16, device=dev)
    ws_r = ft.workspace(ft.route_workspace_size(dsc, T))
    ws_p = ft.workspace(ft.permute_workspace_size(dsc, T))
    ws_a = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    ws_b = ft.workspace(ft.expert_ffn_workspace_size(dsc, T))
    main, side, fill = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    B_P, B_H, host_threads = link_and_host_bandwidth(dev)

    def run(policy, nsteps):
        lru = ft.LRU(1, L.E, C)
        tot.zero_()
        ev_sel, ev_b, ev_a = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(main):
            for i in range(nsteps):
                x = xs[i % len(xs)]
                ft.route(dsc, x, wr, bias, ids, tw, None, ws_r, main)
                ft.permute(dsc, ids, off, sp, pp, ws_p, main)
                lru.step(0, ids, hit, lslot, lev, None, main)
                override = {"qstar": -1, "fill_all": L.k, "fill_none": 0}[policy]
                ft.miss_split(lru, 0, ids, hit, B_P, B_H, override, sa, sb, now, later, cnt, main)
                tot.add_(cnt.to(torch.int64))
                ev_sel.record(main)
                side.wait_event(ev_sel)                       # executor B: the other experts from the host pool
                out_b.zero_()
                ft.expert_ffn(dsc, s_pool, sb, x, off, sp, tw, out_b, ws_b, side)
                ev_b.record(side)
                ft.copy_slots(dsc, s_fill, s_arena, now, cnt[1:2], n, main)   # fills before executor A
                ft.expert_ffn(dsc, s_arena, sa, x, off, sp, None, y_a, ws_a, main)
                main.wait_event(ev_b)
                ft.combine(dsc, T, y_a, pp, tw, ids, sa, out_b, of, ob, main)
                ft.copy_slots(dsc, s_fill, s_arena, later, cnt[2:3], n, main)  # the deferred fills
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        lru.close()
        t = tot.tolist()
        return {"tokens_per_s": round(T * nsteps / dt, 1), "us_per_step": round(dt * 1e6 / nsteps, 2),
                "misses_per_step": round(t[0] / nsteps, 3), "fills_now_per_step": round(t[1] / nsteps, 3),
                "fills_later_per_step": round(t[2] / nsteps, 3), "experts_of_B_per_step": round(t[3] / nsteps, 3)}

    res = {}
    for policy in ("qstar", "fill_all", "fill_none"):
        run(policy, 20)
        res[policy] = run(policy, steps)
    # fill bandwidth: C whole experts from the host pool into the arena, one copy_slots launch
    pairs = torch.stack([torch.arange(C, dtype=torch.int32), torch.arange(C, dtype=torch.int32)], 1).to(dev)
    per_slot = sum(t[0].numel() * t.element_size() for t in (pool.gate, pool.up, pool.down, pool.gate_s, pool.up_s,
                                                             pool.down_s, pool.glob))
    per_slot += ft.prepare_weights_size(dsc, 1)
    ft.copy_slots(dsc, s_fill, s_arena, pairs, None, C, main)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    ft.copy_slots(dsc, s_fill, s_arena, pairs, None, C, main)
    e1.record(main)
    e1.synchronize()
    fill_gbs = C * per_slot / (e0.elapsed_time(e1) / 1e3) / 1e9
    q_mean = res["qstar"]["misses_per_step"]
    return {"workload": f"decode 128x8 d2048 f768 NVFP4, T={T}, slot table C={C} (37%), expert pool in pinned host "
                        f"memory, {steps} steps", "link_gbs": B_P, "host_gbs": B_H, "host_threads": host_threads,
            "qstar_at_mean_misses": round(q_mean * B_P / B_H, 3), "policies": res,
            "fill": {"gbs": round(fill_gbs, 2), "bytes_per_expert": int(per_slot), "experts": C,
                     "of_link": round(fill_gbs / B_P, 3),
                     "how": "one ftmoe_copy_slots launch copying C whole slots (codes, scales, prepared layouts) "
                            "from pinned host memory, CUDA events"},
            "how": "per step: route, permute, LRU, q* split, fills now, executor A (HBM slots) and executor B "
                   "(host pool, side stream), exact merge, deferred fills; wall clock over the steps"}


def stream_leg(layers=3, dev="cuda"):
    """Full-layer double buffering: `layers` prefill layers (128x8, d 2048, f 768, NVFP4) whose
    experts stream from pinned host memory through two device arenas (layer l+1 copied while
    layer l computes) against one arena (the copy waits for the compute), at 4096, 8192 and
    16384 tokens."""
    import sparse_moe_expert_sorted_b300 as ft
    wl = synth.PREFILL
    L = wl.layer
    dsc = ft.desc(L.E, L.k, L.d, L.f, L.fmt, L.renorm)
    Wp = synth.make_experts(L.fmt, layers * L.E, L.d, L.f, 5150, device=dev)
    pin = lambda t: None if t is None else t.cpu().contiguous().pin_memory()
    pool = synth.ExpertWeights(Wp.fmt, Wp.d, Wp.f, pin(Wp.gate), pin(Wp.up), pin(Wp.down), pin(Wp.gate_s),
                               pin(Wp.up_s), pin(Wp.down_s), pin(Wp.glob))
    del Wp
    torch.cuda.empty_cache()
    ft.prepare_weights(dsc, pool)
    z = lambda t: None if t is None else torch.zeros((L.E,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
    arenas = []
    for _ in range(2):
        A = synth.ExpertWeights(pool.fmt, pool.d, pool.f, z(pool.gate), z(pool.up), z(pool.down), z(pool.gate_s),
                                z(pool.up_s), z(pool.down_s), z(pool.glob))
        ft.prepare_weights(dsc, A)
        arenas.append(A)
    structs = [ft.weights_struct(a) for a in arenas]
    routers = [synth.make_router(L.E, L.d, 5160 + l, device=dev) for l in range(layers)]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    out = {}
    for T in (4096, 8192, 16384):
        xs = [synth.make_x(T, L.d, 5170 + l, device=dev) for l in range(layers)]
        of = [torch.empty(T, L.d, device=dev) for _ in range(layers)]
        ws = ft.workspace(ft.layer_workspace_size(dsc, T))
        row = {}
        for n_arenas in (2, 1):
            times = []
            for rep in range(4):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(comp)
                ft.layers_streamed(dsc, ft.weights_struct(pool), structs[:n_arenas], xs, routers, None, of, None, ws,
                                   stream=comp, copy_stream=copy)
                e1.record(comp)
                e1.synchronize()
                if rep:
                    times.append(e0.elapsed_time(e1))
            row[n_arenas] = min(times)
        # the compute alone: the same layers with their experts already resident
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for rep in range(2):
            e0.record(comp)
            for l in range(layers):
                ft.layer_forward(dsc, structs[0], None, xs[l], routers[l], None, None, None, of[l], None, ws, comp)
            e1.record(comp)
            e1.synchronize()
        compute_ms = e0.elapsed_time(e1)
        out[str(T)] = {"ms_two_arenas": round(row[2], 3), "ms_one_arena": round(row[1], 3),
                       "compute_only_ms": round(compute_ms, 3),
                       "tokens_per_s_two_arenas": round(T * layers / (row[2] / 1e3), 1),
                       "penalty_without_second_arena": round(1.0 - row[2] / row[1], 4)}
        del xs, of, ws
    per_layer = sum(t[:L.E].numel() * t.element_size() for t in (pool.gate, pool.up, pool.down, pool.gate_s,
                                                                  pool.up_s, pool.down_s, pool.glob))
    nh = 96 if L.f % 96 == 0 else 64     # the prefill part of the prepared layout (include/ftmoe.h)
    per_layer += L.E * (L.f // nh) * (L.d // 64) * ((2 * nh + 127) // 128) * 512 + L.E * (L.d // 128) * (L.f // 64) * 512
    return {"workload": f"{layers} prefill layers 128x8 d2048 f768 NVFP4, experts in pinned host memory, "
                        "two device arenas vs one", "per_T": out, "bytes_copied_per_layer": int(per_layer),
            "how": "ftmoe_layers_streamed, CUDA events on the compute stream, best of 3 after one warm-up"}


def prefill_leg(args, rank, ws):
    """The metric's second leg: the 8192-token prefill layer (128 experts top-8, d 2048, ffn 768,
    NVFP4), timed like the headline (graph replay between CUDA events, max over ranks), with its
    own FP4 tensor-core roofline, end-to-end figure and CPU baseline."""
    import copy
    pa = copy.copy(args)
    pa.workload, pa.steps, pa.layers, pa.experts = "prefill", args.prefill_steps, 0, 0
    pa.warmup = max(3, min(args.warmup, 5))
    r = bench_ours(pa, rank, ws)
    keys = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "dtype", "config", "roofline", "e2e",
            "gpu_launches", "clocks")
    out = {k: r[k] for k in keys if k in r}
    if rank == 0 and not args.no_cpu_baseline:
        rate, threads, sample, _ = oracle_rate("prefill", args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(rate, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                               "sample": sample}
    return out


def main():
    args = parse()
    if args.steps <= 0:
        args.steps = DEFAULT_STEPS[args.workload]
    if args.impl == "reference":
        # the oracle runs on the host cores of rank 0 only; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(bench_reference(args, 0, 1)), flush=True)
        return
    rank, ws = dist_init()
    res = bench_ours(args, rank, ws)
    if rank == 0 and not args.no_cpu_baseline:
        rate, threads, sample, _ = oracle_rate(args.workload, args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(rate, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                               "sample": sample}
    if args.workload == "decode" and args.prefill_steps > 0 and not args.experts:
        res["prefill_8k"] = prefill_leg(args, rank, ws)
    if args.workload == "decode" and not args.experts and not args.no_cache_legs:
        for key, fn in (("cache", cache_leg), ("stream", stream_leg)):
            try:
                res[key] = fn()
            except Exception as e:   # side reports: never lose the headline line over them
                res[key] = {"error": str(e)[:300]}
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
