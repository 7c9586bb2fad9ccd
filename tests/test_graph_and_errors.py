"""GPU: CUDA-graph replay with nkv advanced on the device ("10 · R4" §2.2:
static grid, nkv as data), the library-owned workspace, and the error paths
that need a device (clamped positions, workspace too small, growth refused
while capturing)."""
import math

import numpy as np
import pytest

import oracle
from harness import assert_close, make_case, run_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import decode_attention_gqa_gb300 as p
    from decode_attention_gqa_gb300 import build
    build.build()
    p.load()
    return p


def test_graph_replay_advances_positions(pkg):
    import torch
    n_head, n_kv, hd, cap = 28, 4, 128, 2048
    scale = 1 / math.sqrt(hd)
    case = make_case(21, 1, n_head, n_kv, hd, cap, (cap,))
    dev = to_device(case)
    P = pkg.attn_split_heuristic(1, n_head, n_kv, hd, cap, 0)
    ws = torch.empty(pkg.attn_workspace_size(1, n_head, hd, P), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(dev["q"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv,
                           hd, scale, cap, n_splits=P, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv,
                           hd, scale, cap, n_splits=P, workspace=ws)
    for nkv in (1, 2, 17, 100, 129, 1000, 2047, 2048):
        dev["positions"].fill_(nkv - 1)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.attn_decode(case["q"], case["k"], case["v"], np.array([nkv - 1], np.int32),
                                 n_head, n_kv, hd, cap, scale)
        assert_close(out.cpu().numpy(), ref, "graph replay nkv=%d" % nkv)


def test_library_owned_workspace_single_sequence(pkg):
    import torch
    n_head, n_kv, hd, cap = 16, 2, 256, 777
    scale = 1 / math.sqrt(hd)
    case = make_case(22, 1, n_head, n_kv, hd, cap, (777,))
    dev = to_device(case)
    out = torch.empty_like(dev["q"])
    pkg.attn_decode(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv, hd, scale)
    torch.cuda.synchronize()
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, scale)
    assert_close(out.cpu().numpy(), ref, "attn_decode")


def test_positions_out_of_range_are_clamped_and_flagged(pkg):
    import torch
    n_head, n_kv, hd, cap = 8, 2, 128, 300
    scale = 1 / math.sqrt(hd)
    case = make_case(23, 3, n_head, n_kv, hd, cap, (300, 300, 300))
    case["positions"] = np.array([cap + 50, -7, 10], np.int32)
    pkg.attn_read_device_error()                               # clear anything stale
    got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale).cpu().numpy()
    flags = pkg.attn_read_device_error()
    assert flags & pkg.ATTN_DEVERR_POSITION_CLAMPED
    assert pkg.attn_read_device_error() == 0                   # cleared by the read
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, scale)
    assert_close(got, ref, "clamped")
    assert np.all(got[1] == 0)
    # in-range positions do not set the flag
    case["positions"] = np.array([cap - 1, 0, 10], np.int32)
    run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale)
    assert pkg.attn_read_device_error() == 0


def test_workspace_errors(pkg):
    import torch
    n_head, n_kv, hd, cap = 8, 2, 128, 256
    scale = 1 / math.sqrt(hd)
    dev = to_device(make_case(24, 1, n_head, n_kv, hd, cap, (200,)))
    out = torch.empty_like(dev["q"])
    need = pkg.attn_workspace_size(1, n_head, hd, 4)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.AttnError) as ei:
        pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv, hd,
                           scale, cap, n_splits=4, workspace=small)
    assert ei.value.status == pkg.ATTN_ERR_WORKSPACE
    # block mode must cover the capacity
    with pytest.raises(pkg.AttnError) as ei:
        pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv, hd,
                           scale, cap, n_splits=2, split_len=64)
    assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG
    # the library-owned workspace may not grow while a stream is capturing
    huge_heads = 64
    qh = torch.zeros(1, huge_heads, hd, device="cuda")
    kh = torch.zeros(1, cap, 8, hd, dtype=torch.float16, device="cuda")
    oh = torch.empty_like(qh)
    lib = pkg.load()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        status = lib.attn_decode_ex(qh.data_ptr(), kh.data_ptr(), kh.data_ptr(),
                                    dev["positions"].data_ptr(), oh.data_ptr(), 1, huge_heads, 8,
                                    hd, scale, cap, 4000, 0, 0, None, 0,
                                    torch.cuda.current_stream().cuda_stream)
    assert status == pkg.ATTN_ERR_WORKSPACE


def test_bounded_wait_runs_out_and_reports(pkg):
    """A wait on an mbarrier nothing arrives on gives up after its limit, sets
    ATTN_DEVERR_PIPELINE_TIMEOUT and returns; the context keeps working."""
    import torch
    pkg.attn_read_device_error()                                  # clear
    s = torch.cuda.Stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        pkg.attn_selftest_bounded_wait(20_000_000, stream=s)      # 20 ms
        e1.record(s)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) >= 19.0                            # it did wait for the limit
    assert pkg.attn_read_device_error(s) == pkg.ATTN_DEVERR_PIPELINE_TIMEOUT
    assert pkg.attn_read_device_error(s) == 0                     # read clears
    # the context still serves a normal call
    n_head, n_kv, hd, cap = 8, 2, 128, 300
    case = make_case(77, 1, n_head, n_kv, hd, cap, (260,))
    got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, 0.1).cpu().numpy()
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, 0.1)
    assert_close(got, ref, "after the self-test")
    assert pkg.attn_read_device_error() == 0
