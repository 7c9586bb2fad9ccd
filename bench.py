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
NOMINAL_HBM_GBS = 7900.0          # GB300 HBM3e data-sheet bandwidth, for context only
KERNEL_SOURCES = ["attn_device.cuh", "attn_partial.cuh", "attn_warp_tc.cuh", "attn_warp_simt.cuh",
                  "attn_warp_tcmq.cuh", "attn_partial_tile.cuh",
                  "attn_partial_umma.cuh", "attn_fused_umma.cuh", "attn_combine.cuh",
                  "attn_kernels_impl.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b", choices=["7b", "long", "stress", "ragged", "tiny"],
                    help="7b (the default bench line) or another workload, for the record")
    ap.add_argument("--ctx", type=int, default=0, help="context override (0 = the workload's)")
    ap.add_argument("--cap", type=int, default=0,
                    help="cache capacity override in rows per sequence (0 = the workload's); "
                         "contexts are clipped to it")
    ap.add_argument("--split-len", type=int, default=0, help="0 = split by count")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--variant", type=int, default=0,
                    help="0 auto, 1 simt, 2 tensor core (mma.sync), 3 tensor core (tcgen05), "
                         "4 tcgen05 with the combine in a thread-block cluster, "
                         "5 one-tile mma.sync")
    ap.add_argument("--splits", type=int, default=0, help="0 = library heuristic")
    ap.add_argument("--kv-dtype", choices=["f16", "bf16"], default="f16")
    ap.add_argument("--append", action="store_true",
                    help="time attn_decode_append (write the new K/V row, then attend)")
    ap.add_argument("--n-q", type=int, default=1,
                    help="causal query rows per sequence (> 1: attn_decode_multi)")
    ap.add_argument("--kv-stable", choices=["on", "off"], default="on",
                    help="flag layers after the first with ATTN_KV_STABLE (their cache and "
                         "positions are not written inside the step)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations the default run records under `workloads`")
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


def strip_comments(src: str) -> str:
    """C++ source without comments and with whitespace collapsed: what the
    compiler sees, so that a comment edit does not count as a kernel change."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_attention_gqa_gb300", "csrc", name)) as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_key(args, w, ctx_end) -> str:
    """The key of a configuration in the profiles/*.md traffic lines: workload,
    context, and every option that changes the kernel or its bytes."""
    key = "%s_ctx%d" % (w.name, ctx_end)
    if args.split_len:
        key += "_blk%d" % args.split_len
    if args.n_q > 1:
        key += "_nq%d" % args.n_q
    if args.kv_dtype != "f16":
        key += "_" + args.kv_dtype
    if args.append:
        key += "_append"
    if args.variant:
        key += "_v%d" % args.variant
    return key


def profiled_traffic(workload_key: str):
    """DRAM read+write bytes per partial launch for a workload from the committed
    ncu summaries (profiles/*.md lines `traffic_per_launch_bytes[<key>]: N`),
    only if the summary's `source_hash` matches the current kernel sources."""
    import glob
    want = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        m_hash = re.search(r"^source_hash:\s*(\w+)", text, re.M)
        m_key = re.search(r"^traffic_per_launch_bytes\[%s\]:\s*(\d+)" % re.escape(workload_key),
                          text, re.M)
        if m_hash and m_key and m_hash.group(1) == want:
            return int(m_key.group(1))
    return None


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

def oracle_sample(layers_host, w, budget_s: float, max_units=None, kv_dtype="f16", n_q=1,
                  threads=None):
    """Run the oracle over (layer, KV head group) units of the workload -- every
    query head of one KV head against that head's rows -- until budget_s (or
    max_units), on `threads` host threads (default: every core the process may
    use); return (GB/s of K+V, units, seconds, threads, what). With n_q > 1 the
    unit holds all n_q causal query rows of the group."""
    import numpy as np
    import oracle
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    G = w.n_head // w.n_kv_head
    units = [(l, hk) for l in range(len(layers_host)) for hk in range(w.n_kv_head)]
    done, nbytes, t0 = 0, 0, time.perf_counter()
    while True:
        l, hk = units[done % len(units)]
        lay = layers_host[l]
        kg = np.ascontiguousarray(lay["k"][:, :, hk:hk + 1])
        vg = np.ascontiguousarray(lay["v"][:, :, hk:hk + 1])
        if n_q > 1:
            qg = np.ascontiguousarray(lay["q"][:, :, hk * G:(hk + 1) * G])
            oracle.attn_decode_multi(qg, kg, vg, lay["positions"], n_q, G, 1, w.head_dim, w.cap,
                                     w.scale, n_threads=threads, kv_dtype=kv_dtype)
        else:
            qg = np.ascontiguousarray(lay["q"][:, hk * G:(hk + 1) * G])
            oracle.attn_decode(qg, kg, vg, lay["positions"], G, 1, w.head_dim, w.cap, w.scale,
                               n_threads=threads, kv_dtype=kv_dtype)
        nbytes += sum(min(max(int(p) + 1, 0), w.cap) for p in lay["positions"]) * w.head_dim * 4
        done += 1
        el = time.perf_counter() - t0
        if max_units is not None:
            if done >= max_units:
                break
        elif el >= budget_s or done >= 100 * len(units):
            break
    what = "%d (layer, KV-head group) units" % done
    return nbytes / el / 1e9, done, el, threads, what


# ------------------------------------------------------------------ our arm

def make_host_layers(w, layers, kv_dtype="f16"):
    from decode_attention_gqa_gb300 import synthetic as syn
    threads = len(os.sched_getaffinity(0))
    return [syn.make_layer(w, layer=l, kv_dtype=kv_dtype, threads=threads) for l in range(layers)]


def config_of(args, w, L, world):
    """The workload as both arms print it: shapes, sizes and mode, nothing
    that depends on the implementation (split count, kernel, flags)."""
    advance = w.n_seq == 1
    ctx_end = max(w.ctx)
    rows = sum(min(max(int(c), 0), w.cap) for c in ([ctx_end] if advance else w.ctx))
    n_q = args.n_q
    extra = "".join([", %d causal query rows per sequence" % n_q if n_q > 1 else "",
                     ", block length %d" % args.split_len if args.split_len else "",
                     ", new K/V row appended by the call" if args.append else ""])
    return {"workload": describe(w, L, args.kv_dtype) + extra,
            "name": w.name, "ctx": ctx_end, "cap": w.cap,
            "n_seq": w.n_seq, "n_head": w.n_head, "n_kv_head": w.n_kv_head,
            "head_dim": w.head_dim, "layers": L, "split_len": args.split_len,
            "kv_dtype": args.kv_dtype, "append": args.append, "n_q": n_q,
            "l2": "inputs larger than L2 (%d MB of K+V per step)"
                  % (rows * w.n_kv_head * w.head_dim * 4 * L // 2 ** 20),
            "parallelism": "replicas" if world > 1 else "single"}


def _t(a):
    """numpy -> torch CPU tensor; bfloat16 bit patterns (uint16) travel as int16."""
    import numpy as np
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)


def workload_for(args):
    from decode_attention_gqa_gb300 import synthetic as syn
    w = syn.WORKLOADS[args.workload]
    if args.ctx:
        w = w.with_ctx(args.ctx)
    if args.cap:
        from dataclasses import replace
        w = replace(w, cap=args.cap, ctx=tuple(min(int(c), args.cap) for c in w.ctx))
    return w


def describe(w, L, kv_dtype="f16"):
    kv = {"f16": "f16", "bf16": "bfloat16"}[kv_dtype]
    return {
        "7b": "7b-like decode: 1 sequence, 28 q / 4 KV heads, head_dim 128, %s KV cache, "
              "%d layers, graph replay with positions += 1 per step" % (kv, L),
        "long": "long-context grouped decode: 1 sequence, 16 q / 2 KV heads, head_dim 256, "
                "context 8400, %s KV cache, %d layers, graph replay with positions += 1 per step"
                % (kv, L),
        "stress": "stress decode: 1 sequence, context 131072, 64 q / 8 KV heads, head_dim 128, "
                  "K x8, %s KV cache, graph replay with positions += 1 per step" % kv,
        "ragged": "batched ragged decode: 32 sequences, context ~ U[1, 32768], 32 q / 8 KV heads, "
                  "head_dim 128, contiguous per-sequence %s KV, static grid" % kv,
        "tiny": "tiny decode: 1 sequence, 8 q / 2 KV heads, head_dim 128, context 512, %s KV cache"
                % kv,
    }.get(w.name, w.name)


# The other configurations a default run records under `workloads`: the long
# grouped layer by count, the fused append and the bfloat16 cache on the 7b
# layer, the long layer at each block length of its sweep, several causal query
# rows, then the stress and ragged calls (the largest caches last: a layer timed
# after their allocations has read up to 5 % slower). Each entry is timed like
# the headline (graph replay, events on the launching stream, its own parity
# spot check against the oracle).
EXTRA_WORKLOADS = [
    ("long", {"workload": "long"}),
    ("7b_append", {"append": True}),
    ("7b_bf16", {"kv_dtype": "bf16"}),
    ("long_blk32", {"workload": "long", "split_len": 32}),
    ("long_blk64", {"workload": "long", "split_len": 64}),
    ("long_blk128", {"workload": "long", "split_len": 128}),
    ("long_blk256", {"workload": "long", "split_len": 256}),
    ("7b_nq2", {"n_q": 2}),
    ("7b_nq4", {"n_q": 4}),
    ("7b_nq8", {"n_q": 8}),
    ("stress", {"workload": "stress"}),
    ("ragged", {"workload": "ragged"}),
]


def is_default_run(args) -> bool:
    return (args.workload == "7b" and not args.ctx and not args.cap and not args.split_len
            and not args.layers and not args.variant and not args.splits and args.kv_dtype == "f16"
            and not args.append and args.n_q == 1 and args.kv_stable == "on")


def summarize(r):
    """One `workloads` entry from a measured line."""
    rf = r["roofline"]
    return {"config": r["config"]["workload"], "kernel": rf["kernel"],
            "partial_variant": rf["partial_variant"], "n_splits": r["plan"]["n_splits"],
            "split_len": r["config"]["split_len"], "us_per_call": r["us_per_layer"],
            "gbs": r["value"], "frac": round(r["value"] / rf["peak"], 4),
            "partial_us": rf["us_per_launch"], "partial_gbs": rf["achieved"],
            "partial_frac": rf["frac"], "combine_us": rf["combine_us_per_launch"],
            "traffic": rf["traffic"], "parity_spot_check": r["parity_spot_check"],
            "steps": r["steps"], "warmup": r["warmup"]}


def run_ours(args, rank, world, local):
    import copy

    import torch

    import decode_attention_gqa_gb300 as pkg
    from decode_attention_gqa_gb300 import build as cuda_build

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    if rank == 0:                        # one build; the other ranks wait for it
        cuda_build.build()
    dist_barrier(world)
    pkg.load()

    line = measure_one(args, rank, world, local)
    if not args.no_workloads and is_default_run(args):
        extra = {}
        for name, over in EXTRA_WORKLOADS:
            a2 = copy.copy(args)
            for k, v in over.items():
                setattr(a2, k, v)
            a2.no_e2e = a2.no_cpu = a2.no_clocks = a2.no_sweep = True
            extra[name] = summarize(measure_one(a2, rank, world, local))
            torch.cuda.empty_cache()
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_one(args, rank, world, local):
    """Time one configuration (the headline, or one `workloads` entry) and
    return its JSON line as a dict."""
    import numpy as np
    import torch

    import decode_attention_gqa_gb300 as pkg
    from decode_attention_gqa_gb300 import build as cuda_build
    from decode_attention_gqa_gb300 import synthetic as syn

    w = workload_for(args)
    L = args.layers or w.layers
    W, K = args.warmup, args.steps
    n_seq = w.n_seq
    advance = n_seq == 1                 # single sequence: nkv grows by one per step
    host = make_host_layers(w, L, args.kv_dtype)
    dev = torch.device("cuda", local)
    s = torch.cuda.Stream(device=dev)
    variant = args.variant | (pkg.ATTN_KV_BF16 if args.kv_dtype == "bf16" else 0)

    n_q = args.n_q
    if n_q > 1:
        if args.append:
            raise SystemExit("--n-q > 1 and --append do not combine (attn_decode_multi has no append)")
        for l, h in enumerate(host):
            h["q"] = syn.make_q_multi(w, n_q, layer=l)
    q = [torch.from_numpy(h["q"]).to(dev) for h in host]
    kc = [_t(h["k"]).to(dev) for h in host]
    vc = [_t(h["v"]).to(dev) for h in host]
    out = [torch.empty_like(x) for x in q]
    pos = torch.from_numpy(host[0]["positions"].copy()).to(dev)
    new_rows = [syn.make_new_rows(w, l, args.kv_dtype) for l in range(L)] if args.append else []
    kn = [_t(r[0]).to(dev) for r in new_rows]
    vn = [_t(r[1]).to(dev) for r in new_rows]
    torch.cuda.synchronize()

    def kv_bytes_for(nkvs):
        return sum(min(max(int(n), 0), w.cap) for n in nkvs) * w.n_kv_head * w.head_dim * 4

    class Plan:
        """Graphs of the L layer calls for one (P, split_len): the whole call, the
        partial stage alone and the combine stage alone."""

        def __init__(self, P, blk):
            self.P, self.blk = P, blk
            self.ws_bytes = pkg.attn_workspace_size(n_seq, n_q * w.n_head, w.head_dim, P)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
            self.g_full = self._capture(advance, "full")
            # the stage entry points serve one query row and keep their partials
            # in the workspace; with n_q > 1, or the cluster-fused kernel (partial
            # and combine in one launch), the whole call stands for the kernel pair
            staged = n_q == 1 and resolved != 4
            self.g_partial = self._capture(False, "partial") if staged else None
            self.g_combine = self._capture(False, "combine") if staged else None

        def _calls(self, stream, stage):
            for l in range(L):
                self.call(l, stream, stage)

        def call(self, l, stream, stage="full"):
            """Layer l's library call on `stream` (the whole call, or one stage)."""
            var = variant | (pkg.ATTN_KV_STABLE if args.kv_stable == "on" and l > 0 else 0)
            if stage == "combine":
                pkg.attn_decode_combine(self.ws, self.ws_bytes, out[l], n_seq, w.n_head,
                                        w.head_dim, self.P, stream=stream)
            elif stage == "partial":
                pkg.attn_decode_partial(q[l], kc[l], vc[l], pos, n_seq, w.n_head, w.n_kv_head,
                                        w.head_dim, w.scale, w.cap, self.P, self.blk,
                                        var, self.ws, self.ws_bytes, stream=stream)
            elif n_q > 1:
                pkg.attn_decode_multi(q[l], kc[l], vc[l], pos, out[l], n_seq, n_q, w.n_head,
                                      w.n_kv_head, w.head_dim, w.scale, w.cap,
                                      n_splits=self.P, split_len=self.blk, variant=var,
                                      workspace=self.ws, workspace_bytes=self.ws_bytes,
                                      stream=stream)
            elif args.append:
                pkg.attn_decode_append(q[l], kn[l], vn[l], kc[l], vc[l], pos, out[l], n_seq,
                                       w.n_head, w.n_kv_head, w.head_dim, w.scale, w.cap,
                                       n_splits=self.P, split_len=self.blk,
                                       variant=var, workspace=self.ws,
                                       workspace_bytes=self.ws_bytes, stream=stream)
            else:
                pkg.attn_decode_ex(q[l], kc[l], vc[l], pos, out[l], n_seq, w.n_head,
                                   w.n_kv_head, w.head_dim, w.scale, w.cap, n_splits=self.P,
                                   split_len=self.blk, variant=var,
                                   workspace=self.ws, workspace_bytes=self.ws_bytes,
                                   stream=stream)

        def _capture(self, adv, stage):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                self._calls(s, stage)              # warm the launch path outside capture
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                if adv:
                    pos.add_(1)
                self._calls(torch.cuda.current_stream(), stage)
            return g

    def timed_replays(g, n, clocks=None, per_step=None):
        """Total ms of n replays (events on the launching stream); with
        per_step a list, also each replay's ms, from one event between replays."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        torch.cuda.synchronize()
        dist_barrier(world)
        if clocks:
            clocks.start()
        with torch.cuda.stream(s):
            ev[0].record(s)
            for i in range(n):
                g.replay()
                if per_step is not None or i == n - 1:
                    ev[i + 1].record(s)
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks else None
        dist_barrier(world)
        if per_step is not None:
            per_step.extend(ev[i].elapsed_time(ev[i + 1]) for i in range(n))
        return ev[0].elapsed_time(ev[n]), clk

    def warm(g):
        with torch.cuda.stream(s):
            for _ in range(W):
                g.replay()

    def measure(plan, ctx_end, clocks=None):
        """Whole-step time and bytes (positions advancing for one sequence), then
        each stage alone at the final nkv. Returns a dict."""
        if advance:
            start = ctx_end - 1 - (W + K)
            assert start >= 0, "context too short for the step count"
            pos.fill_(start)
            nkv_steps = [[start + W + i + 2] for i in range(K)]
        else:
            nkv_steps = [[c for c in w.ctx] for _ in range(K)]
        warm(plan.g_full)
        ms, clk = timed_replays(plan.g_full, K, clocks)
        # the spread from a second pass with an event between replays, so that
        # the events cannot touch the timed total
        steps = []
        if advance:
            pos.fill_(start)
        timed_replays(plan.g_full, K, per_step=steps)
        ms = dist_max(ms, world)
        step_bytes = [kv_bytes_for(n) * L for n in nkv_steps]
        final = nkv_steps[-1]
        if advance:
            pos.fill_(final[0] - 1)
        if plan.g_partial is not None:
            warm(plan.g_partial)
            ms_p, _ = timed_replays(plan.g_partial, K)
            warm(plan.g_combine)
            ms_c, _ = timed_replays(plan.g_combine, K)
        else:
            warm(plan.g_full)
            ms_p, _ = timed_replays(plan.g_full, K)
            ms_c = 0.0
        return {"ms": ms, "clk": clk, "steps_ms": steps, "bytes": sum(step_bytes) * world,
                "partial_us": ms_p * 1e3 / (K * L), "combine_us": ms_c * 1e3 / (K * L),
                "launch_bytes": kv_bytes_for(final)}

    # ---- main timed region: the library's own plan (the split count of the
    # flagged layers 2..L; layer 1 runs the same count without the flag)
    blk0 = args.split_len
    stable_flag = pkg.ATTN_KV_STABLE if args.kv_stable == "on" and L > 1 else 0
    _, P0, _ = pkg.attn_plan_call(n_seq, n_q, w.n_head, w.n_kv_head, w.head_dim, w.cap,
                                  args.splits, blk0, variant | stable_flag)
    # the partial kernel every layer's call runs with that count
    resolved, _, _ = pkg.attn_plan_call(n_seq, n_q, w.n_head, w.n_kv_head, w.head_dim, w.cap, P0,
                                        blk0, variant)
    plan = Plan(P0, blk0)
    launches_per_call = 1 if resolved == 4 else 2       # the cluster-fused kernel has no combine
    ctx_end = max(w.ctx)
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    m0 = measure(plan, ctx_end, clocks)
    value = m0["bytes"] / (m0["ms"] * 1e-3) / 1e9
    us_per_layer = m0["ms"] * 1e3 / (K * L)
    # spread of the timed steps: p10 / median / p90 of each replay's µs per layer
    st = sorted(x * 1e3 / L for x in m0["steps_ms"])
    us_spread = [round(st[int(0.1 * (len(st) - 1))], 3), round(statistics.median(st), 3),
                 round(st[int(0.9 * (len(st) - 1))], 3)] if st else None

    # correctness spot check of layer 0 at the final nkv (oracle). Its inputs
    # are the host copies: for the fused append, layer 0's cache is restored
    # from the host first and the expected cache is built on the host from the
    # original rows and k_new / v_new.
    import oracle
    torch.cuda.synchronize()
    pos_now = pos.cpu().numpy()
    lay0 = dict(host[0], positions=pos_now)
    if args.append:
        kc[0].copy_(_t(host[0]["k"]).to(dev))
        vc[0].copy_(_t(host[0]["v"]).to(dev))
        torch.cuda.synchronize()
        lay0["k"], lay0["v"] = host[0]["k"].copy(), host[0]["v"].copy()
        kn0, vn0 = new_rows[0]
        for si in range(n_seq):
            r = int(pos_now[si])
            if 0 <= r < w.cap:
                lay0["k"][si, r] = kn0[si]
                lay0["v"][si, r] = vn0[si]
    with torch.cuda.stream(s):
        plan._calls(s, "full")
    torch.cuda.synchronize()
    if n_q > 1:
        ref = oracle.attn_decode_multi(lay0["q"], lay0["k"], lay0["v"], lay0["positions"], n_q,
                                       w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale,
                                       n_threads=8, kv_dtype=args.kv_dtype)
        got = out[0].cpu().numpy().astype(np.float64)
        if n_seq > 1:
            ref, got = ref[:3], got[:3]
    elif n_seq == 1:
        ref = oracle.attn_decode(lay0["q"], lay0["k"], lay0["v"], lay0["positions"], w.n_head,
                                 w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=8,
                                 kv_dtype=args.kv_dtype)
        got = out[0].cpu().numpy().astype(np.float64)
    else:
        sidx = [0, n_seq // 2, n_seq - 1]
        ref = np.stack([oracle.attn_decode_one(lay0["q"], lay0["k"], lay0["v"], lay0["positions"],
                                               w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale,
                                               si, 0, kv_dtype=args.kv_dtype) for si in sidx])
        got = out[0].cpu().numpy().astype(np.float64)[sidx, 0]
    parity_ok = bool(np.all(np.abs(got - ref) <= 1e-4 + 1e-3 * np.abs(ref)))

    achieved = m0["launch_bytes"] / (m0["partial_us"] * 1e-6) / 1e9
    peak, peak_kind = measured_peak()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": profiled_traffic(traffic_key(args, w, ctx_end)),
                "kernel": ({4: "attn_fused_umma (partial and combine in one kernel)",
                            3: "attn_split_partial_umma", 5: "attn_split_partial_tile"}
                           .get(resolved, "attn_split_partial"))
                          if n_q == 1 else "attn_split_partial + attn_combine",
                "partial_variant": {1: "simt", 2: "mma.sync", 3: "tcgen05",
                                    4: "tcgen05, cluster-fused",
                                    5: "mma.sync, one tile"}.get(resolved, resolved),
                "bytes_per_launch": m0["launch_bytes"],
                "us_per_launch": round(m0["partial_us"], 3),
                "combine_us_per_launch": round(m0["combine_us"], 3)}

    # ---- sweeps: context (7b) or split block length (long)
    sweep = {}
    if not args.no_sweep:
        if w.name == "7b":
            for c in syn.CTX_SWEEP_7B:
                if c == ctx_end or c > w.cap or c - 1 - (W + K) < 0:
                    continue
                m = measure(plan, c)
                # the plan (kernel and split count) follows the capacity, not the
                # context, so every point runs the headline's kernel
                sweep["ctx%d" % c] = {"partial_variant": roofline["partial_variant"],
                                      "n_splits": plan.P,
                                      "us_per_layer": round(m["ms"] * 1e3 / (K * L), 3),
                                      "gbs": round(m["bytes"] / (m["ms"] * 1e-3) / 1e9, 1),
                                      "partial_us": round(m["partial_us"], 3),
                                      "combine_us": round(m["combine_us"], 3)}
        elif w.name == "long":
            for blk in syn.BLOCK_SWEEP_LONG:
                pb = Plan(-(-w.cap // blk), blk)
                m = measure(pb, ctx_end)
                sweep["blk%d" % blk] = {"n_splits": pb.P,
                                        "us_per_layer": round(m["ms"] * 1e3 / (K * L), 3),
                                        "gbs": round(m["bytes"] / (m["ms"] * 1e-3) / 1e9, 1),
                                        "partial_us": round(m["partial_us"], 3),
                                        "combine_us": round(m["combine_us"], 3)}
                del pb
        if advance:
            pos.fill_(ctx_end - 1)

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        hq = [torch.from_numpy(h["q"]).pin_memory() for h in host]
        hk = [_t(h["k"]).pin_memory() for h in host]
        hv = [_t(h["v"]).pin_memory() for h in host]
        hpos_np = host[0]["positions"].copy()
        if advance:
            hpos_np[:] = ctx_end - 2                    # the graph adds 1
        hpos = torch.from_numpy(hpos_np).pin_memory()
        hout = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in out]
        h2d = sum(t.numel() * t.element_size() for t in hq + hk + hv) + hpos.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in hout)

        # One graph per step: a copy stream brings the inputs layer by layer and
        # layer l's call waits only for its own copies, so the calls (and the
        # read-back of each layer's output) overlap the remaining copies.
        cs = torch.cuda.Stream(device=dev)
        landed = [torch.cuda.Event() for _ in range(L)]
        g_e2e = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g_e2e, stream=s):
            cur = torch.cuda.current_stream()
            cs.wait_stream(cur)
            with torch.cuda.stream(cs):
                pos.copy_(hpos, non_blocking=True)
                for l in range(L):
                    q[l].copy_(hq[l], non_blocking=True)
                    kc[l].copy_(hk[l], non_blocking=True)
                    vc[l].copy_(hv[l], non_blocking=True)
                    landed[l].record(cs)
            for l in range(L):
                cur.wait_event(landed[l])
                if l == 0 and advance:
                    pos.add_(1)
                plan.call(l, cur)
                hout[l].copy_(out[l], non_blocking=True)
            cur.wait_stream(cs)

        def e2e_step():
            with torch.cuda.stream(s):
                g_e2e.replay()

        for _ in range(W):
            e2e_step()
        torch.cuda.synchronize()
        dist_barrier(world)
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        torch.cuda.synchronize()
        el = dist_max(time.perf_counter() - t0, world)
        nkv_e2e = [ctx_end] if advance else list(w.ctx)
        e2e = {"value": round(kv_bytes_for(nkv_e2e) * L * K * world / el / 1e9, 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(el * 1e3 / K, 3)}

    # ---- CPU oracle baseline (rank 0 only, N == 1): on every core the process
    # may use, and on one thread
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, done, el, threads, what = oracle_sample(host, w, budget_s=10.0,
                                                      kv_dtype=args.kv_dtype, n_q=n_q)
        rate1, done1, el1, _, what1 = oracle_sample(host, w, budget_s=8.0, kv_dtype=args.kv_dtype,
                                                    n_q=n_q, threads=1)
        cpu = {"value": round(rate, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%s of the %s workload (%.1f s)" % (what, w.name, el),
               "single_thread": {"value": round(rate1, 4), "unit": UNIT, "cores": 1,
                                 "sample": "%s of the %s workload (%.1f s)" % (what1, w.name, el1)},
               "ms_per_layer_call": round(kv_bytes_for([ctx_end] if advance else w.ctx)
                                          / (rate * 1e9) * 1e3, 3),
               "ms_per_layer_call_single_thread": round(kv_bytes_for([ctx_end] if advance else w.ctx)
                                                        / (rate1 * 1e9) * 1e3, 3)}

    spills = cuda_build.spill_report()
    return {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(m0["ms"] / K, 4),
        "us_per_layer": round(us_per_layer, 3),
        "us_per_layer_p10_p50_p90": us_spread,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(args, w, L, world),
        "plan": {"n_splits": P0, "split_len": blk0, "variant": args.variant,
                 "kv_stable": args.kv_stable, "partial_kernel": roofline["kernel"],
                 "kernels_per_call": launches_per_call},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_call * L * K, "clocks": m0["clk"], "sweep": sweep,
        "parity_spot_check": parity_ok,
        "ptxas_spill_bytes": sum(v["spill_stores"] + v["spill_loads"] for v in spills.values()),
    }


# ------------------------------------------------------- reference arm (oracle)

def run_reference(args, rank, world, local):
    """The oracle timed on the host cores, on this arm's metric and workload;
    each step is a bounded sample -- a few (layer, KV-head group) units -- of
    the step, sized so that warm-up plus steps stay within about two minutes."""
    if rank != 0:
        return
    from decode_attention_gqa_gb300 import synthetic as syn
    w = workload_for(args)
    L = args.layers or w.layers
    host = make_host_layers(w, min(L, 2), args.kv_dtype)
    if args.n_q > 1:
        for l, h in enumerate(host):
            h["q"] = syn.make_q_multi(w, args.n_q, layer=l)
    kw = dict(kv_dtype=args.kv_dtype, n_q=args.n_q)
    rate1, _, el1, threads, _ = oracle_sample(host, w, budget_s=0.0, max_units=1, **kw)
    per_step = max(1, min(L * w.n_kv_head,
                          int(100.0 / max(el1 * (args.steps + args.warmup), 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(host, w, budget_s=0.0, max_units=per_step, **kw)
    total_bytes, total_s = 0.0, 0.0
    for _ in range(args.steps):
        rate, done, el, threads, what = oracle_sample(host, w, budget_s=0.0, max_units=per_step,
                                                      **kw)
        total_bytes += rate * el * 1e9
        total_s += el
    value = total_bytes / total_s / 1e9
    sample = ("%d of the %d (layer, KV-head group) units of a step of the %s workload, per step"
              % (per_step, L * w.n_kv_head, w.name))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(args, w, L, world),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
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
