"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The benchmark runs one independent replica per GPU (no data-path
collective); what it shares across ranks is the barrier around the timed
region and the max over ranks of the elapsed time. Both are exercised here
with world_size 2, as is the rule that only rank 0 prints the reference line.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    try:
        bench.dist_barrier(w)
        got = bench.dist_max(1.5 + rank, w)             # each rank's "elapsed time"
        q.put((r, w, local, got))
        bench.dist_barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[3] == 2.5 for r in res)                # max over ranks, seen by every rank


def test_single_rank_helpers_need_no_process_group(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_max(3.25, 1) == 3.25
    bench.dist_barrier(1)


def test_reference_arm_prints_only_on_rank_zero(capsys):
    import argparse
    import bench
    ns = argparse.Namespace(workload="tiny", ctx=0, layers=0, steps=1, warmup=0, split_len=0)
    bench.run_reference(ns, rank=1, world=2, local=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line_contract():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the keys the benchmark contract names."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                          "--steps", "1", "--warmup", "1"], cwd=root, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"]
    # the same config dict the GPU arm prints for these arguments
    import bench
    old_argv = sys.argv
    try:
        sys.argv = ["bench.py", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
        args = bench.parse_args()
    finally:
        sys.argv = old_argv
    w = bench.workload_for(args)
    assert d["config"] == bench.config_of(args, w, args.layers or w.layers, 1)
