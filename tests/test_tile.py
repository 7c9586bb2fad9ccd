"""GPU parity of the one-tile mma.sync partial kernel (ATTN_VARIANT_TC_TILE:
one tile per block -- 128 rows at head_dim 128, 96 at 256 -- S split by rows
over four warps, one block-wide maximum, O = P·V split by head dimension)
against the double-precision oracle, element by element, through the C ABI.

Covers every group size, both split rules at the chunk boundaries, tiles that
start before the sequence's first row (zero rows from the 4-D tensor map) in a
ragged batch whose unread rows are NaN, large score spread and a planted
dominant row, extreme query magnitudes, bfloat16, the fused append,
early-start chains under graph replay, the 7b and long workloads at full size,
and the argument checks that keep every split within one tile."""
import math

import numpy as np
import pytest

import oracle
from decode_attention_gqa_gb300 import synthetic as syn
from harness import assert_close, make_case, run_decode, to_device
from test_append import _host_after_append, _new_rows, _run_append
from test_kv_stable import _chain

pytestmark = pytest.mark.gpu

VT = 5                       # ATTN_VARIANT_TC_TILE
TILE = {128: 128, 256: 96}   # rows per block


@pytest.fixture(scope="module")
def pkg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import decode_attention_gqa_gb300 as p
    from decode_attention_gqa_gb300 import build
    build.build()
    p.load()
    assert p.ATTN_VARIANT_TC_TILE == VT
    return p


def _oracle(case, n_head, n_kv, hd, cap, scale, kv_dtype="f16"):
    return oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                              hd, cap, scale, n_threads=8, kv_dtype=kv_dtype)


def _check(pkg, case, n_head, n_kv, cap, what, variant=VT, kv_dtype="f16", hd=128, **kw):
    scale = 1 / math.sqrt(hd)
    out = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale, variant=variant, **kw)
    return assert_close(out.cpu().numpy(), _oracle(case, n_head, n_kv, hd, cap, scale, kv_dtype),
                        what)


@pytest.mark.parametrize("hd", [128, 256])
def test_every_group_size(pkg, hd):
    for G in range(1, 9):
        n_kv = 2
        case = make_case(5100 + G + hd, 1, G * n_kv, n_kv, hd, 700, (613,))
        # P * tile >= 700
        for P in ((0, 6, 11) if hd == 128 else (0, 8, 11)):
            _check(pkg, case, G * n_kv, n_kv, 700, "hd%d G%d P=%d" % (hd, G, P), hd=hd, n_splits=P)


@pytest.mark.parametrize("hd", [128, 256])
def test_count_split_boundaries(pkg, hd):
    import torch
    n_head, n_kv, cap = 28, 4, 1024
    P = -(-cap // TILE[hd])                           # chunks of (up to) one tile at full capacity
    base = make_case(5200 + hd, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    dev = to_device(base)
    for nkv in sorted({0, 1, 2, 15, 16, 17, 7, 8, 9, 63, 64, 65, 127, 128, 129, 255, 256, 257,
                       500, 1000, cap - 1, cap}):
        dev["positions"].fill_(nkv - 1)
        out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, n_splits=P, variant=VT)
        ref = _oracle(dict(base, positions=np.array([nkv - 1], np.int32)), n_head, n_kv, hd, cap,
                      scale)
        assert_close(out.cpu().numpy(), ref, "hd%d count split nkv=%d" % (hd, nkv))
        if nkv == 0:
            assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("hd", [128, 256])
def test_block_split_boundaries(pkg, hd):
    n_head, n_kv, cap = 16, 2, 1100
    base = make_case(5300 + hd, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    dev = to_device(base)
    for blk in ((16, 32, 100, 128) if hd == 128 else (16, 32, 64, 96)):
        P = -(-cap // blk)
        for nkv in (1, blk - 1, blk, blk + 1, 3 * blk + 7, cap - 1, cap):
            dev["positions"].fill_(nkv - 1)
            out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, n_splits=P, split_len=blk,
                             variant=VT)
            ref = _oracle(dict(base, positions=np.array([nkv - 1], np.int32)), n_head, n_kv, hd,
                          cap, scale)
            assert_close(out.cpu().numpy(), ref, "hd%d block %d nkv=%d" % (hd, blk, nkv))


def test_balanced_count_split_around_three_quarters_of_a_tile(pkg):
    """By count, a chunk of more than three quarters of a tile is rounded up to
    16 rows, a shorter one to a whole tile: with 76 splits at capacity 8192 the
    rule switches between nkv = 7296 (96-row chunks -> 128) and 7297 (97 -> 112),
    and again at 8513 (113 -> 128; capacity 8704 here). Rows past nkv are NaN."""
    n_head, n_kv, hd, cap, P = 28, 4, 128, 8704, 76
    base = make_case(5350, 1, n_head, n_kv, hd, cap, (cap,))
    for nkv in (1, 1000, 7296, 7297, 7300, 76 * 112, 76 * 112 + 1, 8192, 8600):
        case = dict(base, positions=np.array([nkv - 1], np.int32))
        case["k"] = base["k"].copy()
        case["v"] = base["v"].copy()
        case["k"][0, nkv:] = np.nan
        case["v"][0, nkv:] = np.nan
        _check(pkg, case, n_head, n_kv, cap, "balanced P=76 nkv=%d" % nkv, n_splits=P)


def test_split_count_invariance_and_agreement_with_the_other_kernels(pkg):
    n_head, n_kv, cap = 32, 8, 3000
    case = make_case(5400, 2, n_head, n_kv, 128, cap, (3000, 1234))
    ref = _oracle(case, n_head, n_kv, 128, cap, 1 / math.sqrt(128))
    for P in (24, 25, 32, 64, 188, 400):
        _check(pkg, case, n_head, n_kv, cap, "P=%d" % P, n_splits=P)
    for other in (2, 3):
        got = run_decode(pkg, to_device(case), n_head, n_kv, 128, cap, 1 / math.sqrt(128),
                         n_splits=0, variant=other).cpu().numpy()
        assert_close(got, ref, "variant %d, same inputs" % other)


@pytest.mark.parametrize("hd", [128, 256])
def test_ragged_batch_with_nan_beyond_every_sequence(pkg, hd):
    # sequences after the first start their first tile inside the previous
    # sequence's rows in a flat view; those rows are NaN here
    n_head, n_kv, cap = 32, 8, 900
    ctx = (1, 900, 0, 17, 450, 899, 64, 333, 128, 129)
    case = make_case(5500 + hd, len(ctx), n_head, n_kv, hd, cap, ctx, fill=np.nan)
    for P in ((0, 8, 57) if hd == 128 else (0, 15, 57)):      # P * tile >= 900
        _check(pkg, case, n_head, n_kv, cap, "hd%d ragged P=%d" % (hd, P), hd=hd, n_splits=P)


def test_large_score_spread_and_single_row(pkg):
    n_head, n_kv, cap = 64, 8, 2000
    case = make_case(5600, 1, n_head, n_kv, 128, cap, (1999,), k_scale=8.0)
    case["k"][0, 1234] = (case["k"][0, 1234].astype(np.float32) * 4).astype(np.float16)
    _check(pkg, case, n_head, n_kv, cap, "K x8, planted row")
    one = make_case(5601, 1, 28, 4, 128, 256, (1,), fill=np.nan)
    dev = to_device(one)
    out = run_decode(pkg, dev, 28, 4, 128, 256, 1 / math.sqrt(128), variant=VT).cpu().numpy()
    want = one["v"][0, 0].astype(np.float32)          # [n_kv, hd]
    np.testing.assert_allclose(out[0].reshape(4, 7, 128), np.repeat(want[:, None, :], 7, 1),
                               rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("hd", [128, 256])
def test_extreme_query_magnitudes(pkg, hd):
    # per-head power-of-two scaling of q: no f16 overflow at |q| ~ 1e6 and no
    # loss of the lo part at |q| ~ 1e-6
    n_head, n_kv, cap = 16, 2, 600
    case = make_case(5650 + hd, 1, n_head, n_kv, hd, cap, (555,))
    case["q"][0, :4] *= np.float32(1e6)
    case["q"][0, 4:8] *= np.float32(1e-6)
    case["q"][0, 8] = 0.0
    _check(pkg, case, n_head, n_kv, cap, "hd%d extreme q" % hd, hd=hd)


@pytest.mark.parametrize("hd", [128, 256])
def test_bfloat16_cache(pkg, hd):
    n_head, n_kv, cap = 28, 4, 1500
    case = make_case(5700 + hd, 2, n_head, n_kv, hd, cap, (1500, 700), kv_dtype="bf16")
    _check(pkg, case, n_head, n_kv, cap, "hd%d bf16" % hd, variant=VT | pkg.ATTN_KV_BF16,
           kv_dtype="bf16", hd=hd)


@pytest.mark.parametrize("hd", [128, 256])
def test_fused_append(pkg, hd):
    import torch
    n_kv, G, cap = 2, 7, 300
    n_head = G * n_kv
    scale = 1 / math.sqrt(hd)
    for nkv in (1, 16, 17, 63, 64, 65, 127, 128, 129, 200, cap):
        case = make_case(5800 + nkv + hd, 1, n_head, n_kv, hd, cap, (nkv,))
        case["k"][0, nkv - 1] = np.nan
        case["v"][0, nkv - 1] = np.nan
        k_new, v_new = _new_rows(nkv, 1, n_kv, hd)
        dev = to_device(case)
        kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        for P in (0, 3 if hd == 128 else 5):
            dev = to_device(case)
            got = _run_append(pkg, dev, kn, vn, n_head, n_kv, hd, cap, scale, VT, P)
            kh, vh = _host_after_append(case, k_new, v_new, cap)
            ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap,
                                     scale)
            assert_close(got, ref, "append nkv=%d P=%d" % (nkv, P))
            np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh.view(np.uint16))
            np.testing.assert_array_equal(dev["v"].cpu().numpy().view(np.uint16), vh.view(np.uint16))


@pytest.mark.parametrize("graph, stable", [(False, True), (True, True), (True, False)])
def test_early_start_chain(pkg, graph, stable):
    P = pkg.attn_split_heuristic_ex(1, 1, 28, 4, 128, 2048, 0, VT | pkg.ATTN_KV_STABLE)
    assert P * 128 >= 2048
    _chain(pkg, L=5, n_head=28, n_kv=4, hd=128, cap=2048, ctx=(1900,), P=P, blk=0, variant=VT,
           graph=graph, replays=3, seed=5900, stable=stable)


def test_stable_chain_head_dim_256(pkg):
    P = pkg.attn_split_heuristic_ex(1, 1, 16, 2, 256, 2560, 0, VT | pkg.ATTN_KV_STABLE)
    assert P * TILE[256] >= 2560
    _chain(pkg, L=4, n_head=16, n_kv=2, hd=256, cap=2560, ctx=(1000,), P=P, blk=0, variant=VT,
           graph=True, replays=2, seed=5950)


def test_full_long_workload(pkg):
    w = syn.WORKLOADS["long"]
    lay = syn.make_layer(w)
    P = pkg.attn_split_heuristic_ex(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0,
                                    VT | pkg.ATTN_KV_STABLE)
    assert P * 128 >= w.cap                           # 96-row tiles, or 128-row ones
    v, Pv, _ = pkg.attn_plan_call(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0, 0, 0)
    assert v == VT
    for n in sorted({P, Pv, -(-w.cap // 96)}):
        _check(pkg, lay, w.n_head, w.n_kv_head, w.cap, "long P=%d" % n, hd=w.head_dim, n_splits=n)
    # what variant 0 plans (128-row tiles) at shorter contexts: whole tiles, and half tiles --
    # each block on its last 64 rows -- while the context fits in four tiles
    for ctx in (2048, 513, 512, 300, 65, 64, 1):
        case = dict(lay, positions=np.array([ctx - 1], np.int32))
        _check(pkg, case, w.n_head, w.n_kv_head, w.cap, "long P=%d ctx %d" % (Pv, ctx), hd=w.head_dim,
               n_splits=Pv)


def test_full_7b_workload(pkg):
    w = syn.WORKLOADS["7b"]
    lay = syn.make_layer(w)
    P = pkg.attn_split_heuristic_ex(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0,
                                    VT | pkg.ATTN_KV_STABLE)
    assert P * 128 >= w.cap
    for ctx in syn.CTX_SWEEP_7B:
        case = dict(lay, positions=np.array([ctx - 1], np.int32))
        _check(pkg, case, w.n_head, w.n_kv_head, w.cap, "7b ctx %d" % ctx, n_splits=P)


def test_arguments_that_leave_a_split_larger_than_a_tile(pkg):
    import torch
    case = to_device(make_case(6000, 1, 8, 2, 128, 1024, (1000,)))
    bad = [dict(n_splits=3),                          # 3 * 256 < 1024 (256-row tiles at most)
           dict(n_splits=4, split_len=257),
           dict(n_splits=2, split_len=512)]
    for kw in bad:
        with pytest.raises(pkg.AttnError) as ei:
            run_decode(pkg, case, 8, 2, 128, 1024, 0.1, variant=VT, **kw)
        assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG, kw
    c256 = to_device(make_case(6002, 1, 8, 2, 256, 1024, (1000,)))
    # head_dim 256: 96-row tiles, or 128-row tiles for longer splits, never more
    for kw in (dict(n_splits=7),                                  # 7 * 128 < 1024
               dict(n_splits=8, split_len=129)):
        with pytest.raises(pkg.AttnError) as ei:
            run_decode(pkg, c256, 8, 2, 256, 1024, 0.1, variant=VT, **kw)
        assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG, kw
    # head_dim 64 is not built for this kernel, nor are several query rows at head_dim 256
    c64 = to_device(make_case(6001, 1, 8, 2, 64, 256, (200,)))
    with pytest.raises(pkg.AttnError) as ei:
        run_decode(pkg, c64, 8, 2, 64, 256, 0.1, variant=VT)
    assert ei.value.status == pkg.ATTN_ERR_UNSUPPORTED
    q2 = torch.zeros((1, 2, 8, 256), device="cuda")
    out = torch.empty_like(q2)
    with pytest.raises(pkg.AttnError) as ei:
        pkg.attn_decode_multi(q2, c256["k"], c256["v"], c256["positions"], out, 1, 2, 8, 2, 256,
                              0.1, 1024, n_splits=11, variant=VT)
    assert ei.value.status == pkg.ATTN_ERR_UNSUPPORTED


# ---- several block-length splits per block (split_len divides the tile) ----

@pytest.mark.parametrize("hd,blk", [(128, 16), (128, 32), (128, 64), (256, 16), (256, 32), (256, 48),
                                    (256, 64)])       # 64 at head_dim 256: one split per 96-row tile
def test_several_splits_per_block_with_nan_past_nkv(pkg, hd, blk):
    """One block serves TILE / blk consecutive splits from one tile that starts
    at a multiple of the tile; its rows at or past nkv are read but must never
    reach the result, so they hold NaN here (capacity not a multiple of the tile,
    so the last tile also reaches past the cache)."""
    n_head, n_kv, cap = 14, 2, 1100
    T = TILE[hd]
    base = make_case(6100 + hd + blk, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    P = -(-cap // blk)
    for nkv in sorted({1, 2, blk - 1, blk, blk + 1, T - 1, T, T + 1, 2 * T - blk, 2 * T + 7, 513,
                       cap - T - 1, cap - 1, cap}):
        case = dict(base)
        case["k"] = base["k"].copy()
        case["v"] = base["v"].copy()
        case["k"][0, nkv:] = np.nan
        case["v"][0, nkv:] = np.nan
        case["positions"] = np.array([nkv - 1], np.int32)
        _check(pkg, case, n_head, n_kv, cap, "hd%d blk %d nkv=%d" % (hd, blk, nkv), hd=hd,
               n_splits=P, split_len=blk)


@pytest.mark.parametrize("hd,blk", [(128, 16), (128, 32), (256, 32), (256, 48)])
def test_several_splits_per_block_score_spread(pkg, hd, blk):
    """The splits of a block share one reference maximum, the block's: with K x8
    and a planted row several times larger, the other splits of that block sit
    tens of log2 units below it (their p underflow where they do not matter),
    and a block whose dominant row is in its last split reaches every earlier one."""
    n_head, n_kv, cap = 16, 2, 1000
    case = make_case(6150 + hd + blk, 1, n_head, n_kv, hd, cap, (999,), k_scale=8.0)
    T = TILE[hd]
    for row in (5, 130, 3 * T - 1):                  # a block's first split, a middle one, its last
        case["k"][0, row] = (case["k"][0, row].astype(np.float32) * 4).astype(np.float16)
    _check(pkg, case, n_head, n_kv, cap, "hd%d blk %d spread" % (hd, blk), hd=hd,
           n_splits=-(-cap // blk), split_len=blk)


@pytest.mark.parametrize("hd,blk", [(128, 32), (256, 32), (256, 64)])
def test_several_splits_per_block_ragged_batch(pkg, hd, blk):
    n_head, n_kv, cap = 32, 8, 900
    ctx = (1, 900, 0, 17, 450, 899, 64, 333, 128, 129)
    case = make_case(6200 + hd, len(ctx), n_head, n_kv, hd, cap, ctx, fill=np.nan)
    P = -(-cap // blk)
    for variant in (VT, 0):                       # and whatever variant 0 picks
        _check(pkg, case, n_head, n_kv, cap, "hd%d ragged blk %d variant %d" % (hd, blk, variant),
               hd=hd, n_splits=P, split_len=blk, variant=variant)


@pytest.mark.parametrize("hd", [128, 256])
def test_several_splits_per_block_fused_append(pkg, hd):
    import torch
    n_kv, G, cap, blk = 2, 7, 300, 32
    n_head = G * n_kv
    scale = 1 / math.sqrt(hd)
    P = -(-cap // blk)
    for nkv in (1, 31, 32, 33, 95, 96, 97, 128, 129, 200, cap):
        case = make_case(6300 + nkv + hd, 1, n_head, n_kv, hd, cap, (nkv,))
        case["k"][0, nkv - 1] = np.nan
        case["v"][0, nkv - 1] = np.nan
        k_new, v_new = _new_rows(nkv + 7, 1, n_kv, hd)
        dev = to_device(case)
        kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        out = torch.full_like(dev["q"], float("nan"))
        pkg.attn_decode_append(dev["q"], kn, vn, dev["k"], dev["v"], dev["positions"], out, 1,
                               n_head, n_kv, hd, scale, cap, n_splits=P, split_len=blk, variant=VT)
        torch.cuda.synchronize()
        kh, vh = _host_after_append(case, k_new, v_new, cap)
        ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap, scale)
        assert_close(out.cpu().numpy(), ref, "hd%d append blk %d nkv=%d" % (hd, blk, nkv))
        np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh.view(np.uint16))
        np.testing.assert_array_equal(dev["v"].cpu().numpy().view(np.uint16), vh.view(np.uint16))


def test_several_splits_per_block_stable_chain(pkg):
    _chain(pkg, L=4, n_head=16, n_kv=2, hd=256, cap=2560, ctx=(1000,), P=-(-2560 // 32), blk=32,
           variant=VT, graph=True, replays=2, seed=6400)


def test_full_long_workload_block_32(pkg):
    w = syn.WORKLOADS["long"]
    lay = syn.make_layer(w)
    v, P, _ = pkg.attn_plan_call(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0, 32, 0)
    assert v == VT and P == -(-w.cap // 32)
    _check(pkg, lay, w.n_head, w.n_kv_head, w.cap, "long blk 32", hd=w.head_dim, split_len=32)


# ---- splits of 97..128 rows at head_dim 256: 128-row tiles, one block per SM ----

@pytest.mark.parametrize("hd,G", [(256, 1), (256, 5), (256, 8), (128, 1), (128, 7), (128, 8)])
def test_wide_tile_block_and_count_boundaries(pkg, hd, G):
    """Splits longer than the tile run the wide tile, one block per SM: block
    lengths 97..128 and split counts with 96 P < cap <= 128 P at head_dim 256
    (128-row tiles), block lengths 129..256 and 128 P < cap <= 256 P at 128
    (256-row tiles); every nkv around the split edges, rows past nkv NaN."""
    n_kv, cap = 2, 1100
    W = 128 if hd == 256 else 256                       # the wide tile's rows
    n_head = G * n_kv
    base = make_case(6500 + G + hd, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    if hd == 256:
        cases = ((-(-cap // 128), 128), (-(-cap // 112), 112), (-(-cap // 97), 97), (9, 0), (10, 0), (11, 0))
    else:
        cases = ((-(-cap // 256), 256), (-(-cap // 200), 200), (-(-cap // 129), 129), (5, 0), (6, 0), (8, 0))
    for P, blk in cases:
        v, Pp, _ = pkg.attn_plan_call(1, 1, n_head, n_kv, hd, cap, P, blk, VT)
        assert v == VT and Pp == P
        c = -(-cap // P)                                # by count: near a tile, 16-row chunks
        edge = blk if blk else (-(-c // 16) * 16 if 4 * c > 3 * W else -(-c // W) * W)
        for nkv in (1, edge - 1, edge, edge + 1, 3 * edge + 7, cap - 1, cap):
            case = dict(base, positions=np.array([nkv - 1], np.int32))
            case["k"] = base["k"].copy()
            case["v"] = base["v"].copy()
            case["k"][0, nkv:] = np.nan
            case["v"][0, nkv:] = np.nan
            _check(pkg, case, n_head, n_kv, cap, "G%d P%d blk %d nkv=%d" % (G, P, blk, nkv), hd=hd,
                   n_splits=P, split_len=blk)


def test_wide_tile_ragged_batch_and_automatic_choice(pkg):
    hd, n_head, n_kv, cap, blk = 256, 16, 2, 1000, 128
    ctx = (1, 1000, 0, 127, 128, 129, 500, 999)
    case = make_case(6600, len(ctx), n_head, n_kv, hd, cap, ctx, fill=np.nan)
    v, P, _ = pkg.attn_plan_call(len(ctx), 1, n_head, n_kv, hd, cap, 0, blk, 0)
    assert v == VT and P == -(-cap // blk)
    for variant in (VT, 0, VT | pkg.ATTN_KV_STABLE):
        _check(pkg, case, n_head, n_kv, cap, "wide ragged variant %d" % variant, hd=hd,
               split_len=blk, variant=variant)


def test_wide_tile_fused_append_and_bf16(pkg):
    import torch
    hd, n_kv, G, cap, blk = 256, 2, 8, 300, 128
    n_head = G * n_kv
    scale = 1 / math.sqrt(hd)
    for nkv in (1, 127, 128, 129, 257, cap):
        case = make_case(6700 + nkv, 1, n_head, n_kv, hd, cap, (nkv,))
        k_new, v_new = _new_rows(nkv + 11, 1, n_kv, hd)
        dev = to_device(case)
        kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        out = torch.full_like(dev["q"], float("nan"))
        pkg.attn_decode_append(dev["q"], kn, vn, dev["k"], dev["v"], dev["positions"], out, 1,
                               n_head, n_kv, hd, scale, cap, split_len=blk, variant=VT)
        torch.cuda.synchronize()
        kh, vh = _host_after_append(case, k_new, v_new, cap)
        ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap, scale)
        assert_close(out.cpu().numpy(), ref, "wide append nkv=%d" % nkv)
    for nkv in (5, 200, cap):
        case = make_case(6750 + nkv, 1, n_head, n_kv, hd, cap, (nkv,), kv_dtype="bf16")
        _check(pkg, case, n_head, n_kv, cap, "wide bf16 nkv=%d" % nkv, hd=hd, split_len=blk,
               variant=VT | pkg.ATTN_KV_BF16, kv_dtype="bf16")


def test_wide_tile_stable_chain(pkg):
    _chain(pkg, L=4, n_head=16, n_kv=2, hd=256, cap=2560, ctx=(2000,), P=20, blk=128,
           variant=VT, graph=True, replays=2, seed=6800)


def test_full_7b_workload_on_256_row_tiles(pkg):
    """What variant 0 plans for the 7b layer (256-row tiles, balanced splits),
    at full capacity and shorter contexts -- whole 256-row tiles, and half tiles
    (each block on its last 128 rows) while the context fits in four tiles --
    and block length 256."""
    w = syn.WORKLOADS["7b"]
    lay = syn.make_layer(w)
    v, P, _ = pkg.attn_plan_call(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0, 0, 0)
    assert v == VT and P * 256 >= w.cap
    for ctx in (w.cap, 7777, 2048, 1025, 1024, 1023, 513, 512, 257, 256, 129, 128, 1):
        case = dict(lay, positions=np.array([ctx - 1], np.int32))
        _check(pkg, case, w.n_head, w.n_kv_head, w.cap, "7b P=%d ctx %d" % (P, ctx), n_splits=P)
    _check(pkg, lay, w.n_head, w.n_kv_head, w.cap, "7b blk 256", split_len=256)


@pytest.mark.parametrize("blk", [64, 128])
def test_full_long_workload_block_64_and_128(pkg, blk):
    w = syn.WORKLOADS["long"]
    lay = syn.make_layer(w)
    v, P, _ = pkg.attn_plan_call(1, 1, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0, blk, 0)
    assert v == VT and P == -(-w.cap // blk)
    _check(pkg, lay, w.n_head, w.n_kv_head, w.cap, "long blk %d" % blk, hd=w.head_dim, split_len=blk)


# ---- several causal query rows (head_dim 128, 16 (row, head) slots per block) ----

@pytest.mark.parametrize("n_q", [2, 4])
def test_several_query_rows_full_7b(pkg, n_q):
    """The 7b layer at full size with n_q causal rows per sequence: row i sees
    nkv - n_q + 1 + i cache rows, so the last row of a tile is masked for every
    row but the last (one tile per split)."""
    import torch
    w = syn.WORKLOADS["7b"]
    lay = syn.make_layer(w)
    rng = np.random.Generator(np.random.PCG64([7007, n_q]))
    q = rng.standard_normal((1, n_q, w.n_head, w.head_dim), dtype=np.float32)
    scale = 1 / math.sqrt(w.head_dim)
    # 128-row tiles (64 splits), and 256-row tiles (38 splits: balanced 224-row chunks at
    # full context, whole tiles below 3/4 of a tile, half tiles -- each block on its last
    # 128 rows -- while the context fits in four tiles)
    for P in (w.cap // TILE[128], 38):
        for ctx in (w.cap, 3001, 1000, 200, n_q):
            pos = np.array([ctx - 1], np.int32)
            dev = to_device(dict(lay, q=q, positions=pos))
            out = torch.full_like(dev["q"], float("nan"))
            pkg.attn_decode_multi(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_q, w.n_head,
                                  w.n_kv_head, w.head_dim, scale, w.cap, n_splits=P, variant=VT)
            ref = oracle.attn_decode_multi(q, lay["k"], lay["v"], pos, n_q, w.n_head, w.n_kv_head,
                                           w.head_dim, w.cap, scale, n_threads=8)
            assert_close(out.cpu().numpy(), ref, "7b n_q=%d P=%d ctx %d" % (n_q, P, ctx))


@pytest.mark.parametrize("n_q,G", [(2, 8), (3, 5), (5, 4), (16, 1)])
def test_several_query_rows_nan_past_each_row(pkg, n_q, G):
    """Ragged batch whose cache rows past each sequence's end hold NaN: every
    row's masked positions are read by the tile but must not reach its result."""
    import torch
    n_kv, hd, cap = 2, 128, 700
    n_head = G * n_kv
    ctx = (1, 5, 130, 257, 700)
    case = make_case(7100 + n_q, len(ctx), n_head, n_kv, hd, cap, ctx, fill=float("nan"))
    rng = np.random.Generator(np.random.PCG64([7100, n_q]))
    case["q"] = rng.standard_normal((len(ctx), n_q, n_head, hd), dtype=np.float32)
    scale = 1 / math.sqrt(hd)
    dev = to_device(case)
    for P in (0, 6, 11):
        out = torch.full_like(dev["q"], float("nan"))
        pkg.attn_decode_multi(dev["q"], dev["k"], dev["v"], dev["positions"], out, len(ctx), n_q,
                              n_head, n_kv, hd, scale, cap, n_splits=P, variant=VT)
        ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                       n_head, n_kv, hd, cap, scale, n_threads=8)
        assert_close(out.cpu().numpy(), ref, "n_q=%d G=%d P=%d" % (n_q, G, P))
