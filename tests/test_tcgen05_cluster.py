"""GPU parity of the cluster-fused tcgen05 kernel (ATTN_VARIANT_TCGEN05_CLUSTER:
the 16 splits of a (sequence, KV head) in one thread-block cluster, merged in
distributed shared memory, o written by the kernel; no workspace, no combine
launch) against the double-precision oracle, element by element.

Covers every group size, every number of tiles per block (nkv up to the 8192
the form accepts, with the chunk boundaries), a ragged batch with NaN beyond
every sequence, large score spread, bfloat16, the fused append, early-start
chains under graph replay, the 7b workload at full size, and the argument
checks."""
import math

import numpy as np
import pytest

import oracle
from decode_attention_gqa_gb300 import synthetic as syn
from harness import assert_close, make_case, run_decode, to_device
from test_append import _host_after_append, _new_rows, _run_append
from test_kv_stable import _chain

pytestmark = pytest.mark.gpu

VC = 4                       # ATTN_VARIANT_TCGEN05_CLUSTER


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


def _oracle(case, n_head, n_kv, cap, scale, kv_dtype="f16"):
    return oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                              128, cap, scale, n_threads=8, kv_dtype=kv_dtype)


def _check(pkg, case, n_head, n_kv, cap, what, variant=VC, kv_dtype="f16", **kw):
    scale = 1 / math.sqrt(128)
    out = run_decode(pkg, to_device(case), n_head, n_kv, 128, cap, scale, variant=variant, **kw)
    return assert_close(out.cpu().numpy(), _oracle(case, n_head, n_kv, cap, scale, kv_dtype), what)


def test_every_group_size(pkg):
    for G in range(1, 9):
        n_kv = 2
        case = make_case(5100 + G, 1, G * n_kv, n_kv, 128, 700, (613,))
        for P in (0, 16):
            _check(pkg, case, G * n_kv, n_kv, 700, "G%d P=%d" % (G, P), n_splits=P)


def test_tiles_per_block_and_chunk_boundaries(pkg):
    # chunk = ceil(nkv / 16) rounded up to 128 rows: 1..4 tiles per block
    import torch
    n_head, n_kv, cap = 28, 4, 8192
    base = make_case(5200, 1, n_head, n_kv, 128, cap, (cap,))
    scale = 1 / math.sqrt(128)
    dev = to_device(base)
    for nkv in (0, 1, 2, 127, 128, 129, 2047, 2048, 2049, 2050, 4095, 4096, 4097, 6000, 6143,
                6144, 6145, 8000, 8191, 8192):
        dev["positions"].fill_(nkv - 1)
        out = run_decode(pkg, dev, n_head, n_kv, 128, cap, scale, variant=VC)
        ref = _oracle(dict(base, positions=np.array([nkv - 1], np.int32)), n_head, n_kv, cap, scale)
        assert_close(out.cpu().numpy(), ref, "nkv=%d" % nkv)
        if nkv == 0:
            assert torch.count_nonzero(out).item() == 0


def test_ragged_batch_with_nan_beyond_every_sequence(pkg):
    n_head, n_kv, cap = 32, 8, 2000
    ctx = (1, 2000, 0, 17, 450, 1999, 64, 333, 128, 129, 1025)
    case = make_case(5300, len(ctx), n_head, n_kv, 128, cap, ctx, fill=np.nan)
    _check(pkg, case, n_head, n_kv, cap, "ragged")


def test_large_score_spread_and_bfloat16(pkg):
    n_head, n_kv, cap = 64, 8, 4000
    case = make_case(5400, 1, n_head, n_kv, 128, cap, (3999,), k_scale=8.0)
    case["k"][0, 1234] = (case["k"][0, 1234].astype(np.float32) * 4).astype(np.float16)
    _check(pkg, case, n_head, n_kv, cap, "K x8, planted row")
    b = make_case(5401, 2, 28, 4, 128, 3000, (3000, 700), kv_dtype="bf16")
    _check(pkg, b, 28, 4, 3000, "bf16", variant=VC | pkg.ATTN_KV_BF16, kv_dtype="bf16")


def test_fused_append(pkg):
    import torch
    n_kv, G, cap = 2, 7, 3000
    n_head = G * n_kv
    scale = 1 / math.sqrt(128)
    for nkv in (1, 127, 128, 129, 2048, 2049, 2999, cap):
        case = make_case(5500 + nkv, 1, n_head, n_kv, 128, cap, (nkv,))
        case["k"][0, nkv - 1] = np.nan
        case["v"][0, nkv - 1] = np.nan
        k_new, v_new = _new_rows(nkv, 1, n_kv, 128)
        dev = to_device(case)
        kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        got = _run_append(pkg, dev, kn, vn, n_head, n_kv, 128, cap, scale, VC, 0)
        kh, vh = _host_after_append(case, k_new, v_new, cap)
        ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, 128, cap, scale)
        assert_close(got, ref, "append nkv=%d" % nkv)
        np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh.view(np.uint16))
        np.testing.assert_array_equal(dev["v"].cpu().numpy().view(np.uint16), vh.view(np.uint16))


@pytest.mark.parametrize("graph, stable", [(False, True), (True, True), (True, False)])
def test_early_start_chain(pkg, graph, stable):
    _chain(pkg, L=5, n_head=28, n_kv=4, hd=128, cap=4096, ctx=(3900,), P=16, blk=0, variant=VC,
           graph=graph, replays=3, seed=5600, stable=stable)


def test_full_7b_workload(pkg):
    w = syn.WORKLOADS["7b"]
    lay = syn.make_layer(w)
    for ctx in syn.CTX_SWEEP_7B:
        case = dict(lay, positions=np.array([ctx - 1], np.int32))
        _check(pkg, case, w.n_head, w.n_kv_head, w.cap, "7b ctx %d" % ctx)


def test_arguments_outside_the_fused_form(pkg):
    import torch
    case = to_device(make_case(5700, 1, 8, 2, 128, 1024, (1000,)))
    for kw in (dict(n_splits=8), dict(n_splits=32), dict(n_splits=8, split_len=128)):
        with pytest.raises(pkg.AttnError) as ei:
            run_decode(pkg, case, 8, 2, 128, 1024, 0.1, variant=VC, **kw)
        assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG, kw
    big = to_device(make_case(5701, 1, 8, 2, 128, 8193, (8000,)))
    with pytest.raises(pkg.AttnError) as ei:
        run_decode(pkg, big, 8, 2, 128, 8193, 0.1, variant=VC)
    assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG
    c256 = to_device(make_case(5702, 1, 8, 2, 256, 512, (500,)))
    with pytest.raises(pkg.AttnError) as ei:
        run_decode(pkg, c256, 8, 2, 256, 512, 0.1, variant=VC)
    assert ei.value.status == pkg.ATTN_ERR_UNSUPPORTED
    # the stage entry points keep their partials in a workspace: not this form
    ws_bytes = pkg.attn_workspace_size(1, 8, 128, 16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.AttnError) as ei:
        pkg.attn_decode_partial(case["q"], case["k"], case["v"], case["positions"], 1, 8, 2, 128, 0.1,
                                1024, 16, 0, VC, ws, ws_bytes)
    assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG
