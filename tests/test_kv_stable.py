"""GPU: ATTN_KV_STABLE (early start). Layers after the first read positions and
start their K/V copies before the previous kernel on the stream has ended;
q, k_new and the workspace must still wait for it. The chains below make any
early read of those visible: layer l + 1 takes the previous layer's output as
its q (written by the combine kernel just before it, NaN until then), and all
layers share one workspace (the flagged partial kernel overwrites what the
previous combine reads). The expected values are the oracle's own chain, with
its f32-rounded output as the next layer's q."""
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


def _oracle_chain(q0, layers, positions, n_head, n_kv, hd, cap, scale, kv_dtype="f16"):
    outs, q = [], q0
    for lay in layers:
        o = oracle.attn_decode(q, lay["k"], lay["v"], positions, n_head, n_kv, hd, cap, scale,
                               n_threads=8, kv_dtype=kv_dtype)
        outs.append(o)
        q = o.astype(np.float32)
    return outs


def _chain(pkg, L, n_head, n_kv, hd, cap, ctx, P, blk, variant, graph, replays, seed, stable=True):
    import torch
    n_seq = len(ctx)
    layers = [make_case(seed + l, n_seq, n_head, n_kv, hd, cap, ctx) for l in range(L)]
    dev = [to_device(c) for c in layers]
    q0 = torch.from_numpy(layers[0]["q"]).cuda()
    pos = torch.from_numpy(layers[0]["positions"] - 1).cuda()      # the step adds 1
    outs = [torch.empty_like(q0) for _ in range(L)]
    scale = 1 / math.sqrt(hd)
    P = P or pkg.attn_split_heuristic(n_seq, n_head, n_kv, hd, cap, 0)
    ws_bytes = pkg.attn_workspace_size(n_seq, n_head, hd, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    pkg.attn_read_device_error()                     # clear what earlier tests left

    def step():
        pos.add_(1)
        for l in range(L):
            var = variant | (pkg.ATTN_KV_STABLE if stable and l > 0 else 0)
            pkg.attn_decode_ex(q0 if l == 0 else outs[l - 1], dev[l]["k"], dev[l]["v"], pos,
                               outs[l], n_seq, n_head, n_kv, hd, scale, cap, n_splits=P,
                               split_len=blk, variant=var, workspace=ws, workspace_bytes=ws_bytes,
                               stream=s)

    g = None
    if graph:
        with torch.cuda.stream(s):
            step()                                   # uncaptured warm-up of the launch path
        torch.cuda.synchronize()
        pos.sub_(1)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        torch.cuda.synchronize()
    for r in range(replays):
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        if graph:
            with torch.cuda.stream(s):
                g.replay()
        else:
            with torch.cuda.stream(s):
                step()
        torch.cuda.synchronize()
        positions = pos.cpu().numpy()
        ref = _oracle_chain(layers[0]["q"], layers, positions, n_head, n_kv, hd, cap, scale)
        for l in range(L):
            assert_close(outs[l].cpu().numpy(), ref[l], "layer %d replay %d" % (l, r))
    flags = pkg.attn_read_device_error()
    assert flags == 0


@pytest.mark.parametrize("graph, stable", [(False, True), (True, True), (True, False)])
def test_stable_chain_7b_shape(pkg, graph, stable):
    # stable=False: the same chain without the flag (every read after the wait)
    _chain(pkg, L=5, n_head=28, n_kv=4, hd=128, cap=2048, ctx=(1900,), P=0, blk=0, variant=0,
           graph=graph, replays=3, seed=900, stable=stable)


@pytest.mark.parametrize("P, blk", [(1, 0), (19, 0), (40, 64)])
def test_stable_chain_split_choices(pkg, P, blk):
    # P = 40 with 64-row blocks at nkv ~ 1000: the later splits are empty
    _chain(pkg, L=4, n_head=16, n_kv=2, hd=256, cap=2560, ctx=(1000,), P=P, blk=blk, variant=0,
           graph=True, replays=2, seed=910)


@pytest.mark.parametrize("variant", [1, 2])
def test_stable_chain_ragged_batch(pkg, variant):
    _chain(pkg, L=3, n_head=32, n_kv=8, hd=128, cap=700, ctx=(1, 699, 17, 450, 0, 333),
           P=0, blk=0, variant=variant, graph=True, replays=2, seed=920)


def test_stable_append_chain(pkg):
    """Flagged appends: the new row still comes from k_new / v_new, which the
    kernel reads only after the wait."""
    import torch
    L, n_head, n_kv, hd, cap, nkv = 3, 28, 4, 128, 1024, 777
    layers = [make_case(930 + l, 1, n_head, n_kv, hd, cap, (nkv,)) for l in range(L)]
    dev = [to_device(c) for c in layers]
    rng = np.random.Generator(np.random.PCG64(931))
    kn = [rng.standard_normal((1, n_kv, hd), dtype=np.float32).astype(np.float16) for _ in range(L)]
    vn = [rng.standard_normal((1, n_kv, hd), dtype=np.float32).astype(np.float16) for _ in range(L)]
    kn_d = [torch.from_numpy(x).cuda() for x in kn]
    vn_d = [torch.from_numpy(x).cuda() for x in vn]
    q0 = torch.from_numpy(layers[0]["q"]).cuda()
    pos = torch.from_numpy(layers[0]["positions"]).cuda()
    outs = [torch.full_like(q0, float("nan")) for _ in range(L)]
    P = 24
    ws_bytes = pkg.attn_workspace_size(1, n_head, hd, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for l in range(L):
            pkg.attn_decode_append(q0 if l == 0 else outs[l - 1], kn_d[l], vn_d[l], dev[l]["k"],
                                   dev[l]["v"], pos, outs[l], 1, n_head, n_kv, hd, 1 / math.sqrt(hd),
                                   cap, n_splits=P, variant=pkg.ATTN_KV_STABLE if l else 0,
                                   workspace=ws, workspace_bytes=ws_bytes, stream=s)
    torch.cuda.synchronize()
    for l in range(L):
        layers[l]["k"][0, nkv - 1] = kn[l][0]
        layers[l]["v"][0, nkv - 1] = vn[l][0]
    ref = _oracle_chain(layers[0]["q"], layers, layers[0]["positions"], n_head, n_kv, hd, cap,
                        1 / math.sqrt(hd))
    for l in range(L):
        assert_close(outs[l].cpu().numpy(), ref[l], "append layer %d" % l)
        np.testing.assert_array_equal(dev[l]["k"].cpu().numpy(), layers[l]["k"])


def test_stable_flag_accepted_with_every_entry_point(pkg):
    import torch
    n_head, n_kv, hd, cap = 8, 2, 128, 300
    case = make_case(940, 1, n_head, n_kv, hd, cap, (250,))
    d = to_device(case)
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, 0.1)
    out = torch.full_like(d["q"], float("nan"))
    pkg.attn_decode_static(d["q"], d["k"], d["v"], d["positions"], out, 1, n_head, n_kv, hd, 0.1,
                           cap, variant=pkg.ATTN_KV_STABLE)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "static + stable")
    qm = torch.from_numpy(np.repeat(case["q"][:, None], 2, axis=1)).cuda()
    outm = torch.full_like(qm, float("nan"))
    pkg.attn_decode_multi(qm, d["k"], d["v"], d["positions"], outm, 1, 2, n_head, n_kv, hd, 0.1,
                          cap, variant=pkg.ATTN_KV_STABLE)
    torch.cuda.synchronize()
    assert_close(outm.cpu().numpy()[:, 1], ref, "multi + stable, last query row")


# ------------------------------------- full size, in the launch configuration bench.py times

def _bench_configuration(pkg, name, L, n_q=1, variant=0):
    """L independent layers of a workload at full size in one captured graph:
    positions += 1, then layer 0 without and layers 1.. with ATTN_KV_STABLE,
    split count from attn_split_heuristic_ex for that flag -- the step bench.py
    times. Every layer is compared with the oracle after one replay."""
    import torch
    from decode_attention_gqa_gb300 import synthetic as syn
    w = syn.WORKLOADS[name]
    layers = [syn.make_layer(w, layer=l) for l in range(L)]
    if n_q > 1:
        for l, lay in enumerate(layers):
            lay["q"] = syn.make_q_multi(w, n_q, layer=l)
    dev = [to_device(c) for c in layers]
    pos = torch.from_numpy(layers[0]["positions"] - 1).cuda()
    outs = [torch.full_like(d["q"], float("nan")) for d in dev]
    P = pkg.attn_split_heuristic_ex(w.n_seq, n_q, w.n_head, w.n_kv_head, w.head_dim, w.cap, 0,
                                    variant | pkg.ATTN_KV_STABLE)
    ws_bytes = pkg.attn_workspace_size(w.n_seq, n_q * w.n_head, w.head_dim, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        pos.add_(1)
        for l in range(L):
            var = variant | (pkg.ATTN_KV_STABLE if l > 0 else 0)
            if n_q > 1:
                pkg.attn_decode_multi(dev[l]["q"], dev[l]["k"], dev[l]["v"], pos, outs[l], w.n_seq,
                                      n_q, w.n_head, w.n_kv_head, w.head_dim, w.scale, w.cap,
                                      n_splits=P, variant=var, workspace=ws,
                                      workspace_bytes=ws_bytes, stream=s)
            else:
                pkg.attn_decode_ex(dev[l]["q"], dev[l]["k"], dev[l]["v"], pos, outs[l], w.n_seq,
                                   w.n_head, w.n_kv_head, w.head_dim, w.scale, w.cap, n_splits=P,
                                   variant=var, workspace=ws, workspace_bytes=ws_bytes, stream=s)

    with torch.cuda.stream(s):
        step()                                        # warm the launch path
    torch.cuda.synchronize()
    pos.sub_(1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    positions = pos.cpu().numpy()
    assert np.array_equal(positions, layers[0]["positions"])
    for l in range(L):
        lay = layers[l]
        if n_q > 1:
            ref = oracle.attn_decode_multi(lay["q"], lay["k"], lay["v"], positions, n_q, w.n_head,
                                           w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=16)
        else:
            ref = oracle.attn_decode(lay["q"], lay["k"], lay["v"], positions, w.n_head,
                                     w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=16)
        assert_close(outs[l].cpu().numpy(), ref, "%s n_q=%d layer %d (P=%d)" % (name, n_q, l, P))
    assert pkg.attn_read_device_error() == 0
    return P


def torch_sm_count():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_full_7b_bench_configuration(pkg):
    # variant 0 runs this short call on the one-tile kernel: 256-row tiles, one block per
    # SM, 38 splits of 216 -> 224 rows on 152 SMs (128-row tiles, 64, where one block per
    # SM would leave chunks of 192 rows or fewer)
    P = _bench_configuration(pkg, "7b", L=4)
    P1 = torch_sm_count() // 4
    c1 = -(-8192 // P1)
    assert P == (P1 if 192 < c1 <= 256 else 64)
    assert _bench_configuration(pkg, "7b", L=3, variant=pkg.ATTN_VARIANT_TC_TILE) == 64
    # the mma.sync kernel at its own split count (blocks of its three-tile ring)
    assert _bench_configuration(pkg, "7b", L=3, variant=pkg.ATTN_VARIANT_TC) == 43


def test_full_long_bench_configuration(pkg):
    # variant 0 runs the one-tile kernel at head_dim 256 too: 128-row tiles, one block per
    # SM, 76 splits of 111 -> 112 rows on 152 SMs (whole 96-row tiles, 88, where one
    # block per SM would leave chunks of 96 rows or fewer)
    P = _bench_configuration(pkg, "long", L=3)
    P1 = torch_sm_count() // 2
    c1 = -(-8400 // P1)
    assert P == (P1 if 96 < c1 <= 128 else 88)
    assert _bench_configuration(pkg, "long", L=3, variant=pkg.ATTN_VARIANT_TC_TILE) == 88
    assert _bench_configuration(pkg, "long", L=2, variant=pkg.ATTN_VARIANT_TC) == 75


def test_full_7b_four_query_rows_bench_configuration(pkg):
    _bench_configuration(pkg, "7b", L=3, n_q=4)
