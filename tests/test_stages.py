"""GPU: the two stages as separate calls (attn_decode_partial, then
attn_decode_combine) and the documented workspace layout.

The layout test emulates sharding the KV rows of one sequence across two
devices: each part of the cache gets its own partial call, the two
workspaces' splits are laid side by side along the split axis (the exchange
a multi-device run would do with an all-gather), and one combine call must
give the oracle's attention over the whole cache."""
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


def _stages(pkg, dev, n_seq, n_head, n_kv, hd, cap, scale, P, blk=0, variant=0):
    import torch
    ws_bytes = pkg.attn_workspace_size(n_seq, n_head, hd, P)
    ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full_like(dev["q"], float("nan"))
    pkg.attn_decode_partial(dev["q"], dev["k"], dev["v"], dev["positions"], n_seq, n_head, n_kv,
                            hd, scale, cap, P, blk, variant, ws, ws_bytes)
    pkg.attn_decode_combine(ws, ws_bytes, out, n_seq, n_head, hd, P)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ws


@pytest.mark.parametrize("hd, variant", [(128, 0), (128, 1), (256, 1), (256, 2), (64, 2), (8, 1)])
def test_partial_then_combine(pkg, hd, variant):
    n_head, n_kv, cap = 8, 2, 700
    ctx = (650, 1, 0, 333)
    case = make_case(1100 + hd + variant, len(ctx), n_head, n_kv, hd, cap, ctx)
    scale = 1 / math.sqrt(hd)
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, scale, n_threads=8)
    for P, blk in ((7, 0), (12, 64), (64, 0), (70, 16)):
        got, _ = _stages(pkg, to_device(case), len(ctx), n_head, n_kv, hd, cap, scale, P, blk,
                         variant)
        assert_close(got, ref, "stages hd%d variant %d P=%d blk=%d" % (hd, variant, P, blk))


def _halves(ws, n_seq, n_head, hd, P):
    """(oc, ml) views of a workspace per the documented layout."""
    N = P
    flat = ws.cpu().numpy().view(np.float32)
    o_floats = n_seq * n_head * N * hd
    ml_off = (o_floats * 4 + 255) // 256 * 256 // 4
    oc = flat[:o_floats].reshape(n_seq, n_head, N, hd)
    ml = flat[ml_off:ml_off + n_seq * n_head * N * 2].reshape(n_seq, n_head, N, 2)
    return oc, ml


@pytest.mark.parametrize("variant", [0, 1])
def test_splits_of_two_row_shards_combine_like_one_call(pkg, variant):
    import torch
    n_head, n_kv, hd, n = 28, 4, 128, 1500
    half = 640                                   # shard A: rows [0, 640), shard B: [640, 1500)
    case = make_case(1200 + variant, 1, n_head, n_kv, hd, n, (n,))
    scale = 1 / math.sqrt(hd)
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             n, scale, n_threads=8)
    shards = []
    for lo, hi, P in ((0, half, 5), (half, n, 9)):
        sub = dict(case, k=np.ascontiguousarray(case["k"][:, lo:hi]),
                   v=np.ascontiguousarray(case["v"][:, lo:hi]),
                   positions=np.array([hi - lo - 1], dtype=np.int32))
        _, ws = _stages(pkg, to_device(sub), 1, n_head, n_kv, hd, hi - lo, scale, P, 0, variant)
        shards.append((_halves(ws, 1, n_head, hd, P), P))
    # the exchange: splits side by side along the split axis
    (oca, mla), Pa = shards[0]
    (ocb, mlb), Pb = shards[1]
    P = Pa + Pb
    ws_bytes = pkg.attn_workspace_size(1, n_head, hd, P)
    oc = np.concatenate([oca, ocb], axis=2)
    ml = np.concatenate([mla, mlb], axis=2)
    buf = np.full(ws_bytes // 4, np.nan, dtype=np.float32)
    o_floats = oc.size
    ml_off = (o_floats * 4 + 255) // 256 * 256 // 4
    buf[:o_floats] = oc.ravel()
    buf[ml_off:ml_off + ml.size] = ml.ravel()
    ws = torch.from_numpy(buf).cuda()
    out = torch.full((1, n_head, hd), float("nan"), device="cuda")
    pkg.attn_decode_combine(ws, ws_bytes, out, 1, n_head, hd, P)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "two shards variant %d" % variant)
    # and the splits of an empty shard change nothing (their oc is never read)
    ml2 = np.concatenate([ml, np.tile(np.array([-np.inf, 0], np.float32), (1, n_head, 3, 1))],
                         axis=2)
    oc2 = np.concatenate([oc, np.full((1, n_head, 3, hd), np.nan, np.float32)], axis=2)
    ws_bytes2 = pkg.attn_workspace_size(1, n_head, hd, P + 3)
    buf2 = np.full(ws_bytes2 // 4, np.nan, dtype=np.float32)
    ml_off2 = (oc2.size * 4 + 255) // 256 * 256 // 4
    buf2[:oc2.size] = oc2.ravel()
    buf2[ml_off2:ml_off2 + ml2.size] = ml2.ravel()
    out2 = torch.full_like(out, float("nan"))
    pkg.attn_decode_combine(torch.from_numpy(buf2).cuda(), ws_bytes2, out2, 1, n_head, hd, P + 3)
    torch.cuda.synchronize()
    assert_close(out2.cpu().numpy(), ref, "two shards + an empty one")


def test_every_split_empty_gives_zero(pkg):
    import torch
    n_head, hd, P = 4, 128, 3
    ws_bytes = pkg.attn_workspace_size(2, n_head, hd, P)
    buf = np.full(ws_bytes // 4, np.nan, dtype=np.float32)
    N = P
    o_floats = 2 * n_head * N * hd
    ml_off = (o_floats * 4 + 255) // 256 * 256 // 4
    buf[ml_off:ml_off + 2 * n_head * N * 2] = np.tile([-np.inf, 0.0], 2 * n_head * N)
    out = torch.full((2, n_head, hd), float("nan"), device="cuda")
    pkg.attn_decode_combine(torch.from_numpy(buf).cuda(), ws_bytes, out, 2, n_head, hd, P)
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == 0.0)
