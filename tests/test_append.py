"""GPU: fused KV append (attn_decode_append) -- the new token's K/V row is
written into cache row positions[s] and attended in the same launches
(dotLLM #199 §1: write the new row, then attend over [0, nkv)).

Checked against the oracle run on a host copy of the cache with the new row
written, with the device cache's old content at that row set to NaN (so any
read of the stale row would show), plus a bit-exact check of the cache after
the call, out-of-range positions, several sequences and a graph replay that
appends one row per step.
"""
import math

import numpy as np
import pytest

import oracle
from harness import assert_close, make_case, to_device

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


def _new_rows(seed, n_seq, n_kv, hd):
    rng = np.random.Generator(np.random.PCG64([seed, 77]))
    k = rng.standard_normal((n_seq, n_kv, hd), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((n_seq, n_kv, hd), dtype=np.float32).astype(np.float16)
    return k, v


def _host_after_append(case, k_new, v_new, cap):
    k, v = case["k"].copy(), case["v"].copy()
    for s, p in enumerate(case["positions"]):
        if 0 <= p < cap:
            k[s, p] = k_new[s]
            v[s, p] = v_new[s]
    return k, v


def _run_append(pkg, dev, kn, vn, n_head, n_kv, hd, cap, scale, variant, P=0):
    import torch
    out = torch.full_like(dev["q"], float("nan"))
    pkg.attn_decode_append(dev["q"], kn, vn, dev["k"], dev["v"], dev["positions"], out,
                           dev["positions"].shape[0], n_head, n_kv, hd, scale, cap, n_splits=P,
                           variant=variant)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("variant,hd,G", [(2, 128, 7), (2, 256, 8), (2, 64, 4), (1, 128, 4),
                                          (1, 8, 2), (1, 256, 8)])
def test_append_then_attend(pkg, variant, hd, G):
    import torch
    n_kv, cap = 2, 300
    n_head = G * n_kv
    scale = 1 / math.sqrt(hd)
    for nkv in (1, 16, 17, 64, 65, 129, 200, cap):
        case = make_case(40 + nkv, 1, n_head, n_kv, hd, cap, (nkv,))
        case["k"][0, nkv - 1] = np.nan            # stale content of the row to be written
        case["v"][0, nkv - 1] = np.nan
        k_new, v_new = _new_rows(nkv, 1, n_kv, hd)
        dev = to_device(case)
        kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        for P in (0, 3):
            got = _run_append(pkg, dev, kn, vn, n_head, n_kv, hd, cap, scale, variant, P)
            kh, vh = _host_after_append(case, k_new, v_new, cap)
            ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap,
                                     scale)
            assert_close(got, ref, "append nkv=%d P=%d" % (nkv, P))
            # the cache now holds the new row; every other row is untouched
            np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16),
                                          kh.view(np.uint16))
            np.testing.assert_array_equal(dev["v"].cpu().numpy().view(np.uint16),
                                          vh.view(np.uint16))


@pytest.mark.parametrize("variant", [1, 2])
def test_append_several_sequences_and_bad_positions(pkg, variant):
    import torch
    n_head, n_kv, hd, cap = 32, 8, 128, 500
    ctx = (1, 500, 37, 250, 0, 499)
    case = make_case(50, len(ctx), n_head, n_kv, hd, cap, ctx)
    case["positions"] = np.array([0, 499, 36, 249, -1, 700], np.int32)   # last one out of range
    k_new, v_new = _new_rows(5, len(ctx), n_kv, hd)
    dev = to_device(case)
    kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
    pkg.attn_read_device_error()
    got = _run_append(pkg, dev, kn, vn, n_head, n_kv, hd, cap, 1 / math.sqrt(hd), variant)
    assert pkg.attn_read_device_error() & pkg.ATTN_DEVERR_POSITION_CLAMPED
    kh, vh = _host_after_append(case, k_new, v_new, cap)
    ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap,
                             1 / math.sqrt(hd))
    assert_close(got, ref, "append batch")
    np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh.view(np.uint16))
    np.testing.assert_array_equal(dev["v"].cpu().numpy().view(np.uint16), vh.view(np.uint16))
    assert np.all(got[4] == 0)


def test_append_graph_replay_one_row_per_step(pkg):
    import torch
    n_head, n_kv, hd, cap = 28, 4, 128, 1024
    scale = 1 / math.sqrt(hd)
    start = 700
    case = make_case(60, 1, n_head, n_kv, hd, cap, (start,))
    dev = to_device(case)
    kn = torch.zeros(1, n_kv, hd, dtype=torch.float16, device="cuda")
    vn = torch.zeros_like(kn)
    P = pkg.attn_split_heuristic(1, n_head, n_kv, hd, cap, 0)
    ws = torch.empty(pkg.attn_workspace_size(1, n_head, hd, P), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(dev["q"])

    def call():
        pkg.attn_decode_append(dev["q"], kn, vn, dev["k"], dev["v"], dev["positions"], out, 1,
                               n_head, n_kv, hd, scale, cap, n_splits=P, workspace=ws)

    dev["positions"].fill_(start - 1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()                                   # rewrites row start-1 with zeros
    torch.cuda.synchronize()
    kh, vh = case["k"].copy(), case["v"].copy()
    kh[0, start - 1] = 0
    vh[0, start - 1] = 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dev["positions"].add_(1)
        call()
    for step in range(4):
        k_new, v_new = _new_rows(100 + step, 1, n_kv, hd)
        kn.copy_(torch.from_numpy(k_new))
        vn.copy_(torch.from_numpy(v_new))
        g.replay()
        torch.cuda.synchronize()
        p = start + step
        kh[0, p], vh[0, p] = k_new[0], v_new[0]
        ref = oracle.attn_decode(case["q"], kh, vh, np.array([p], np.int32), n_head, n_kv, hd, cap,
                                 scale)
        assert_close(out.cpu().numpy(), ref, "graph append step %d" % step)
    np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh.view(np.uint16))
