#!/usr/bin/env python3
"""Benchmark: split-KV grouped-query decode attention on GB300.

A step is one decode step of the 7B-like workload: 28 independent layers, each
one call of the library (partial + combine kernels) over its own q and f16 KV
cache (1 sequence, 28 query / 4 KV heads, head_dim 128), captured once in a
CUDA graph that first advances nkv on the device (positions += 1) -- the
static-grid, nkv-as-data replay of minfer "10 · R4" §2.2. The 28 caches
(470 MB at context 8192) are larger than L2, so no flush is needed between
steps.

Printed: one JSON line (rank 0) with the metric
  "decode-attn µs/layer and achieved HBM GB/s (K+V bytes/time) vs GB300 peak"
where value = K+V bytes of rows [0, nkv) read per step, all ranks, / time.
Extra keys: µs per layer, a context sweep, the roofline of the partial kernel
(timed alone in a graph of partial-only launches), the end-to-end number
through the C ABI from pinned host buffers, the CPU oracle baseline, clocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/layer and achieved HBM GB/s (K+V bytes/time) vs GB300 peak"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["attn_device.cuh", "attn_partial.cuh", "attn_combine.cuh",
                  "attn_kernels_impl.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b", choices=["7b"])
    ap.add_argument("--ctx", type=int, default=8192)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--variant", type=int, default=0, help="0 auto, 1 simt, 2 tensor core")
    ap.add_argument("--splits", type=int, default=0, help="0 = library heuristic")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend, init_method="env://")


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_attention_gqa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_key: str):
    """DRAM bytes per partial launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "attn_split_partial_7b_ctx8192.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"^source_hash:\s*(\w+)", text, re.M)
    m_key = re.search(r"^traffic_per_launch_bytes\[%s\]:\s*(\d+)" % re.escape(workload_key), text, re.M)
    if not m_hash or not m_key or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_key.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.proc = None
        self.enabled = enabled
        self.path = os.path.join("/tmp", "attn_bench_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        if not self.enabled:
            return
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle leg

def oracle_rate(layers_host, w, ctx, budget_s: float, max_layers=None):
    """Run the oracle (all host cores) over layers until budget_s; return
    (GB/s of K+V, layers done, seconds, threads)."""
    import oracle
    threads = len(os.sched_getaffinity(0))
    bytes_per_layer = ctx * w.n_kv_head * w.head_dim * 4
    done, t0 = 0, time.perf_counter()
    n = len(layers_host) if max_layers is None else max_layers
    while True:
        lay = layers_host[done % len(layers_host)]
        oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head, w.n_kv_head,
                           w.head_dim, w.cap, w.scale, n_threads=threads)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= n:
            break
    return done * bytes_per_layer / el / 1e9, done, el, threads


# ------------------------------------------------------------------ our arm

def make_host_layers(w, ctx, layers):
    from decode_attention_gqa_gb300 import synthetic as syn
    wc = w.with_ctx(ctx)
    out = []
    for l in range(layers):
        lay = syn.make_layer(wc, layer=l)
        out.append(lay)
    return wc, out


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import decode_attention_gqa_gb300 as pkg
    from decode_attention_gqa_gb300 import build as cuda_build
    from decode_attention_gqa_gb300 import synthetic as syn

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    if rank == 0 or not os.path.exists(pkg.library_path()):
        cuda_build.build()
    dist_barrier(world)
    pkg.load()

    w = syn.WORKLOADS[args.workload]
    L = args.layers or w.layers
    ctx_end = args.ctx
    W, K = args.warmup, args.steps
    wc, host = make_host_layers(w, ctx_end, L)
    dev = torch.device("cuda", local)
    s = torch.cuda.Stream(device=dev)

    # device copies: every layer its own q, K, V, out; one positions array
    q = [torch.from_numpy(h["q"]).to(dev) for h in host]
    kc = [torch.from_numpy(h["k"]).to(dev) for h in host]
    vc = [torch.from_numpy(h["v"]).to(dev) for h in host]
    out = [torch.empty_like(x) for x in q]
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    P = args.splits or pkg.attn_split_heuristic(1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0)
    ws_bytes = pkg.attn_workspace_size(1, w.n_head, w.head_dim, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def layer_calls(stream, partial_only=False, combine_only=False):
        for l in range(L):
            if combine_only:
                pkg.attn_decode_combine(ws, ws_bytes, out[l], 1, w.n_head, w.head_dim, P,
                                        stream=stream)
            elif partial_only:
                pkg.attn_decode_partial(q[l], kc[l], vc[l], pos, 1, w.n_head, w.n_kv_head,
                                        w.head_dim, w.scale, w.cap, P, 0, args.variant, ws,
                                        ws_bytes, stream=stream)
            else:
                pkg.attn_decode_ex(q[l], kc[l], vc[l], pos, out[l], 1, w.n_head, w.n_kv_head,
                                   w.head_dim, w.scale, w.cap, n_splits=P, variant=args.variant,
                                   workspace=ws, workspace_bytes=ws_bytes, stream=stream)

    def capture(advance: bool, partial_only=False, combine_only=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            layer_calls(s, partial_only, combine_only)   # warm the launch path outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            if advance:
                pos.add_(1)
            layer_calls(torch.cuda.current_stream(), partial_only, combine_only)
        return g

    def timed_replays(g, n, clocks=None):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        dist_barrier(world)
        if clocks:
            clocks.start()
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(n):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks else None
        dist_barrier(world)
        return e0.elapsed_time(e1), clk

    def kv_bytes(nkv):
        return nkv * w.n_kv_head * w.head_dim * 2 * 2

    # ---- main timed region: W warm-up + K timed replays of the 28-layer step
    g = capture(advance=True)
    start_pos = ctx_end - 1 - (W + K)
    assert start_pos >= 0, "context too short for the step count"
    pos.fill_(start_pos)
    with torch.cuda.stream(s):
        for _ in range(W):
            g.replay()
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    ms, clk = timed_replays(g, K, clocks)
    nkvs = [start_pos + W + i + 2 for i in range(K)]        # nkv seen by timed step i
    step_bytes = [kv_bytes(n) * L for n in nkvs]
    ms_max = dist_max(ms, world)
    total_bytes = sum(step_bytes) * world
    value = total_bytes / (ms_max * 1e-3) / 1e9
    us_per_layer = ms_max * 1e3 / (K * L)

    # correctness spot check of the last step (oracle, one layer)
    import oracle
    lay0 = dict(host[0], positions=np.array([nkvs[-1] - 1], np.int32))
    ref = oracle.attn_decode(lay0["q"], lay0["k"], lay0["v"], lay0["positions"], w.n_head,
                             w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=8)
    got = out[0].cpu().numpy().astype(np.float64)
    parity_ok = bool(np.all(np.abs(got - ref) <= 1e-4 + 1e-3 * np.abs(ref)))

    # ---- each stage alone: graphs of L partial-only and L combine-only launches
    gp = capture(advance=False, partial_only=True)
    gc = capture(advance=False, combine_only=True)

    def stage_times(c):
        """(partial µs, combine µs) per launch at nkv = c."""
        pos.fill_(c - 1)
        with torch.cuda.stream(s):
            for _ in range(W):
                gp.replay()
        ms_p, _ = timed_replays(gp, K)
        with torch.cuda.stream(s):
            for _ in range(W):
                gc.replay()
        ms_c, _ = timed_replays(gc, K)
        return ms_p * 1e3 / (K * L), ms_c * 1e3 / (K * L)

    partial_us, combine_us = stage_times(ctx_end)
    achieved = kv_bytes(ctx_end) / (partial_us * 1e-6) / 1e9
    peak, peak_kind = measured_peak()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": profiled_traffic("7b_ctx%d" % ctx_end),
                "kernel": "attn_split_partial", "bytes_per_launch": kv_bytes(ctx_end),
                "us_per_launch": round(partial_us, 3), "combine_us_per_launch": round(combine_us, 3)}

    # ---- context sweep (same caches, positions set per point)
    sweep = {}
    if not args.no_sweep:
        for c in syn.CTX_SWEEP_7B:
            if c == ctx_end or c - 1 - (W + K) < 0:
                continue
            pos.fill_(c - 1 - (W + K))
            with torch.cuda.stream(s):
                for _ in range(W):
                    g.replay()
            ms_c, _ = timed_replays(g, K)
            ms_c = dist_max(ms_c, world)
            b = sum(kv_bytes(c - K + i + 1) * L for i in range(K))
            p_us, c_us = stage_times(c)
            sweep[str(c)] = {"us_per_layer": round(ms_c * 1e3 / (K * L), 3),
                             "gbs": round(b * world / (ms_c * 1e-3) / 1e9, 1),
                             "partial_us": round(p_us, 3), "combine_us": round(c_us, 3)}
    pos.fill_(ctx_end - 1)

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        hq = [torch.from_numpy(h["q"]).pin_memory() for h in host]
        hk = [torch.from_numpy(h["k"]).pin_memory() for h in host]
        hv = [torch.from_numpy(h["v"]).pin_memory() for h in host]
        hpos = torch.tensor([ctx_end - 2], dtype=torch.int32).pin_memory()   # +1 in the graph
        hout = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in out]
        h2d = sum(t.numel() * t.element_size() for t in hq + hk + hv) + 4
        d2h = sum(t.numel() * t.element_size() for t in hout)

        def e2e_step():
            with torch.cuda.stream(s):
                pos.copy_(hpos, non_blocking=True)
                for l in range(L):
                    q[l].copy_(hq[l], non_blocking=True)
                    kc[l].copy_(hk[l], non_blocking=True)
                    vc[l].copy_(hv[l], non_blocking=True)
                g.replay()
                for l in range(L):
                    hout[l].copy_(out[l], non_blocking=True)

        for _ in range(W):
            e2e_step()
        torch.cuda.synchronize()
        dist_barrier(world)
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        torch.cuda.synchronize()
        el = dist_max(time.perf_counter() - t0, world)
        e2e = {"value": round(kv_bytes(ctx_end) * L * K * world / el / 1e9, 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(el * 1e3 / K, 3)}

    # ---- CPU oracle baseline (rank 0 only, N == 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, done, el, threads = oracle_rate(host, wc, ctx_end, budget_s=10.0, max_layers=10 * L)
        cpu = {"value": round(rate, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d layer calls of the %s workload at context %d (%.1f s)"
                         % (done, args.workload, ctx_end, el)}

    spills = cuda_build.spill_report()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_max / K, 4),
            "us_per_layer": round(us_per_layer, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "7b-like decode: 1 sequence, 28 q / 4 KV heads, head_dim 128, "
                                   "f16 KV cache, %d layers, graph replay with positions += 1 "
                                   "per step" % L,
                       "ctx": ctx_end, "cap": w.cap, "n_head": w.n_head, "n_kv_head": w.n_kv_head,
                       "head_dim": w.head_dim, "layers": L, "n_splits": P,
                       "variant": args.variant, "kv_dtype": "f16",
                       "l2": "inputs larger than L2 (%d MB of K+V per step)"
                             % (kv_bytes(ctx_end) * L // 2 ** 20),
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 2 * L * K, "clocks": clk, "sweep": sweep,
            "parity_last_step": parity_ok,
            "ptxas_spill_bytes": sum(v["spill_stores"] + v["spill_loads"] for v in spills.values()),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- reference arm (oracle)

def run_reference(args, rank, world, local):
    """The oracle timed on the host cores, on this arm's metric and workload;
    each step is a bounded sample (a few layer calls) of the step."""
    if rank != 0:
        return
    from decode_attention_gqa_gb300 import synthetic as syn
    w = syn.WORKLOADS[args.workload]
    L = args.layers or w.layers
    ctx = args.ctx
    wc, host = make_host_layers(w, ctx, min(L, 4))
    bytes_per_layer = ctx * w.n_kv_head * w.head_dim * 4
    threads = len(os.sched_getaffinity(0))
    # size a step so that warmup + steps stay within about two minutes
    _, _, el1, _ = oracle_rate(host, wc, ctx, budget_s=0.0, max_layers=1)
    per_step_layers = max(1, min(L, int(4.0 / max(el1, 1e-6))))
    per_step_layers = min(per_step_layers, max(1, int(100.0 / max(el1 * (args.steps + args.warmup), 1e-6))))
    for _ in range(args.warmup):
        oracle_rate(host, wc, ctx, budget_s=0.0, max_layers=per_step_layers)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rate(host, wc, ctx, budget_s=0.0, max_layers=per_step_layers)
    el = time.perf_counter() - t0
    value = per_step_layers * args.steps * bytes_per_layer / el / 1e9
    sample = ("%d of %d layer calls per step of the %s workload at context %d"
              % (per_step_layers, L, args.workload, ctx))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3),
        "us_per_layer": round(el * 1e6 / (args.steps * per_step_layers), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "7b-like decode: 1 sequence, 28 q / 4 KV heads, head_dim 128, "
                               "f16 KV cache, %d layers" % L, "ctx": ctx, "layers": L},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
