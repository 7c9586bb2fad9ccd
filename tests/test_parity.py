"""GPU parity: the CUDA path through the C ABI against the double-precision
oracle, element by element, on seeded inputs.

Covers every compiled (head_dim, group) pair, both split rules at the chunk
boundaries that make splits empty ("10 · R4" §4: nkv at multiples of the chunk
and their neighbours), ragged multi-sequence batches, NaN in unread rows,
split-count invariance, large score spread, and every workload at its full
size in the launch configuration the benchmark times (sampled outputs where
the oracle would be slow).
"""
import math

import numpy as np
import pytest

import oracle
from decode_attention_gqa_gb300 import synthetic as syn
from harness import assert_close, make_case, run_decode, to_device

pytestmark = pytest.mark.gpu

VARIANTS = [1, 2]       # ATTN_VARIANT_SIMT (CUDA cores), ATTN_VARIANT_TC (tensor cores)


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


def _oracle(case, n_head, n_kv, hd, cap, scale, threads=8):
    return oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                              hd, cap, scale, n_threads=threads)


def _check(pkg, case, n_head, n_kv, hd, cap, scale, what, **kw):
    dev = to_device(case)
    out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, **kw)
    got = out.cpu().numpy()
    ref = _oracle(case, n_head, n_kv, hd, cap, scale)
    return assert_close(got, ref, what)


# ------------------------------------------------------------ the workloads

def test_tiny_workload(pkg):
    w = syn.WORKLOADS["tiny"]
    lay = syn.make_layer(w)
    _check(pkg, lay, w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale, "tiny", n_splits=w.n_splits)


def test_smallhead_fixture(pkg):
    w = syn.WORKLOADS["smallhead"]
    lay = syn.make_layer(w)
    for P in (0, 1, 4):
        _check(pkg, lay, w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale, "smallhead P=%d" % P,
               n_splits=P)


# ------------------------------------------------------ every compiled shape

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("hd", [8, 64, 128, 256])
def test_all_groups_and_head_dims(pkg, hd, variant):
    if variant == 2 and hd % 16:
        pytest.skip("the tensor-core kernel needs head_dim % 16 == 0")
    for G in range(1, 9):
        n_kv = 2
        n_head = G * n_kv
        cap = 700
        case = make_case(100 * hd + G, 1, n_head, n_kv, hd, cap, (613,))
        _check(pkg, case, n_head, n_kv, hd, cap, 1 / math.sqrt(hd), "hd%d G%d" % (hd, G),
               n_splits=5, variant=variant)


# --------------------------------------------------- split boundaries (R4 §4)

@pytest.mark.parametrize("variant", VARIANTS)
def test_count_split_boundaries(pkg, variant):
    n_head, n_kv, hd, cap, P = 28, 4, 128, 1024, 8
    base = make_case(7, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    dev = to_device(base)
    import torch
    nkvs = sorted({0, 1, 2, 15, 16, 17, P - 1, P, P + 1, 31, 32, 33, 127, 128, 129, 255, 256, 257,
                   16 * P - 1, 16 * P, 16 * P + 1, 500, cap - 1, cap})
    for nkv in nkvs:
        dev["positions"].fill_(nkv - 1)
        out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, n_splits=P, variant=variant)
        case = dict(base, positions=np.array([nkv - 1], np.int32))
        ref = _oracle(case, n_head, n_kv, hd, cap, scale)
        assert_close(out.cpu().numpy(), ref, "count split nkv=%d" % nkv)
        if nkv == 0:
            assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_split_boundaries(pkg, variant):
    n_head, n_kv, hd, cap = 16, 2, 256, 1100
    base = make_case(8, 1, n_head, n_kv, hd, cap, (cap,))
    scale = 1 / math.sqrt(hd)
    dev = to_device(base)
    for blk in (32, 64, 128, 256, 100):
        P = -(-cap // blk)
        for nkv in (1, blk - 1, blk, blk + 1, 3 * blk, 3 * blk + 7, cap - 1, cap):
            dev["positions"].fill_(nkv - 1)
            out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, n_splits=P, split_len=blk,
                             variant=variant)
            case = dict(base, positions=np.array([nkv - 1], np.int32))
            ref = _oracle(case, n_head, n_kv, hd, cap, scale)
            assert_close(out.cpu().numpy(), ref, "block %d nkv=%d" % (blk, nkv))


@pytest.mark.parametrize("variant", VARIANTS)
def test_split_count_invariance(pkg, variant):
    n_head, n_kv, hd, cap = 32, 8, 128, 3000
    case = make_case(9, 2, n_head, n_kv, hd, cap, (3000, 1234))
    scale = 1 / math.sqrt(hd)
    ref = _oracle(case, n_head, n_kv, hd, cap, scale)
    dev = to_device(case)
    outs = []
    for P in (1, 2, 3, 7, 32, 33, 63, 64, 65, 188, 400):
        out = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, n_splits=P, variant=variant)
        outs.append(out.cpu().numpy())
        assert_close(outs[-1], ref, "P=%d" % P)


# ------------------------------------------------------------ ragged batch

@pytest.mark.parametrize("variant", VARIANTS)
def test_ragged_multisequence_with_nan_tail(pkg, variant):
    n_head, n_kv, hd, cap = 32, 8, 128, 900
    ctx = (1, 900, 0, 17, 450, 899, 64, 333)
    case = make_case(10, len(ctx), n_head, n_kv, hd, cap, ctx, fill=np.nan)
    scale = 1 / math.sqrt(hd)
    for P, blk in ((0, 0), (4, 0), (15, 64)):
        got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale, n_splits=P,
                         split_len=blk, variant=variant).cpu().numpy()
        assert np.all(np.isfinite(got))
        ref = _oracle(case, n_head, n_kv, hd, cap, scale)
        assert_close(got, ref, "ragged P=%d blk=%d" % (P, blk))
        assert np.all(got[2] == 0)                       # empty sequence -> 0


# ----------------------------------------------------------- numerics

@pytest.mark.parametrize("variant", VARIANTS)
def test_large_score_spread_and_planted_row(pkg, variant):
    n_head, n_kv, hd, cap = 64, 8, 128, 20000
    case = make_case(11, 1, n_head, n_kv, hd, cap, (cap,), k_scale=8.0)
    scale = 1 / math.sqrt(hd)
    _check(pkg, case, n_head, n_kv, hd, cap, scale, "K x8", variant=variant)
    # a row aligned with every query of KV head 3 takes all the weight
    j = 12345
    q = case["q"]
    q[0, 24:32] = q[0, 24]
    case["k"][0, j, 3] = (q[0, 24] * 40).astype(np.float16)
    dev = to_device(case)
    got = run_decode(pkg, dev, n_head, n_kv, hd, cap, scale, variant=variant).cpu().numpy()
    want = case["v"][0, j, 3].astype(np.float64)
    for h in range(24, 32):
        assert_close(got[0, h], want, "planted row head %d" % h)


@pytest.mark.parametrize("variant", VARIANTS)
def test_single_row_is_that_v_row(pkg, variant):
    n_head, n_kv, hd, cap = 8, 2, 128, 64
    case = make_case(12, 1, n_head, n_kv, hd, cap, (1,))
    got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, 0.3,
                     variant=variant).cpu().numpy()
    for h in range(n_head):
        np.testing.assert_array_equal(got[0, h], case["v"][0, 0, h // 4].astype(np.float32))


@pytest.mark.parametrize("variant", VARIANTS)
def test_extreme_query_magnitudes(pkg, variant):
    """q rows scaled by 1e-30 .. 1e4 (outside f16 range): the tensor-core kernel's
    per-head power-of-two scaling keeps them finite and accurate."""
    n_head, n_kv, hd, cap = 8, 2, 128, 300
    case = make_case(13, 1, n_head, n_kv, hd, cap, (300,))
    case["q"][0, 0] *= 1e-30
    case["q"][0, 1] *= 1e-3
    case["q"][0, 2] *= 30.0
    case["q"][0, 5, :64] *= 1e4
    _check(pkg, case, n_head, n_kv, hd, cap, 1 / math.sqrt(hd), "extreme q", variant=variant)


# ------------------------------------------ full-size workloads, bench config

def _full_workload(pkg, name, sample_pairs=None, threads=16):
    w = syn.WORKLOADS[name]
    lay = syn.make_layer(w)
    dev = to_device(lay)
    kw = {}
    if w.split_len:
        kw = dict(n_splits=-(-w.cap // w.split_len), split_len=w.split_len)
    gots = {}
    for variant in (0,) + tuple(VARIANTS):
        gots[variant] = run_decode(pkg, dev, w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale,
                                   variant=variant, **kw).cpu().numpy()
    del dev
    if sample_pairs is None:
        ref = oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                                 w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=threads)
        for variant, got in gots.items():
            assert_close(got, ref, "%s variant %d" % (name, variant))
        return
    for (s, h) in sample_pairs:
        ref = oracle.attn_decode_one(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                                     w.n_kv_head, w.head_dim, w.cap, w.scale, s, h)
        for variant, got in gots.items():
            assert_close(got[s, h], ref, "%s variant %d s=%d h=%d" % (name, variant, s, h))


def test_full_7b_all_contexts(pkg):
    w = syn.WORKLOADS["7b"]
    for ctx in syn.CTX_SWEEP_7B:
        wc = w.with_ctx(ctx)
        lay = syn.make_layer(wc)
        dev = to_device(lay)
        ref = oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], wc.n_head,
                                 wc.n_kv_head, wc.head_dim, wc.cap, wc.scale, n_threads=16)
        for variant in (0,) + tuple(VARIANTS):
            got = run_decode(pkg, dev, wc.n_head, wc.n_kv_head, wc.head_dim, wc.cap, wc.scale,
                             variant=variant).cpu().numpy()
            assert_close(got, ref, "7b ctx=%d variant %d" % (ctx, variant))


def test_full_long_grouped_all_blocks(pkg):
    w = syn.WORKLOADS["long"]
    lay = syn.make_layer(w)
    dev = to_device(lay)
    ref = oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                             w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=16)
    for blk in syn.BLOCK_SWEEP_LONG:
        for variant in (0,) + tuple(VARIANTS):
            got = run_decode(pkg, dev, w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale,
                             n_splits=-(-w.cap // blk), split_len=blk,
                             variant=variant).cpu().numpy()
            assert_close(got, ref, "long blk=%d variant %d" % (blk, variant))


def test_full_stress(pkg):
    _full_workload(pkg, "stress")


def test_full_ragged_sampled(pkg):
    w = syn.WORKLOADS["ragged"]
    rng = np.random.Generator(np.random.PCG64(77))
    pairs = [(s, int(rng.integers(0, w.n_head))) for s in range(w.n_seq)]
    _full_workload(pkg, "ragged", sample_pairs=pairs)


# ------------------------------------------------------------ grid extremes

@pytest.mark.parametrize("variant", VARIANTS)
def test_grid_z_at_its_limit(pkg, variant):
    """65535 sequences (the largest grid z) of 0 to 2 rows each, every one
    checked against the oracle."""
    n_seq, n_head, n_kv, hd, cap = 65535, 8, 2, 64, 2
    rng = np.random.Generator(np.random.PCG64(1400))
    ctx = tuple(int(c) for c in rng.integers(0, cap + 1, n_seq))
    case = make_case(1401, n_seq, n_head, n_kv, hd, cap, ctx)
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, 0.125, n_threads=16)
    got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, 0.125, variant=variant)
    assert_close(got.cpu().numpy(), ref, "65535 sequences variant %d" % variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_largest_split_count(pkg, variant):
    """P = 4096 (the most the library takes): by count most splits are empty;
    by 1-row blocks every row is a split of its own."""
    n_head, n_kv, hd, cap = 8, 2, 128, 4096
    case = make_case(1402, 2, n_head, n_kv, hd, cap, (4096, 1999))
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, 0.09, n_threads=16)
    dev = to_device(case)
    for blk in (0, 1):
        got = run_decode(pkg, dev, n_head, n_kv, hd, cap, 0.09, n_splits=4096, split_len=blk,
                         variant=variant)
        assert_close(got.cpu().numpy(), ref, "P=4096 blk=%d variant %d" % (blk, variant))


@pytest.mark.parametrize("kv", ["f16", "bf16"])
def test_decode_attention_convenience_call(pkg, kv):
    """decode_attention infers the sizes from the tensors and picks the cache
    type; one and several query rows."""
    import torch
    n_head, n_kv, hd, cap = 28, 4, 128, 900
    case = make_case(1500, 2, n_head, n_kv, hd, cap, (900, 321), kv_dtype=kv)
    dev = to_device(case)
    if kv == "bf16":
        dev["k"], dev["v"] = dev["k"].view(torch.bfloat16), dev["v"].view(torch.bfloat16)
    out = pkg.decode_attention(dev["q"], dev["k"], dev["v"], dev["positions"])
    torch.cuda.synchronize()
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, 1 / math.sqrt(hd), n_threads=8, kv_dtype=kv)
    assert_close(out.cpu().numpy(), ref, "decode_attention %s" % kv)
    rng = np.random.Generator(np.random.PCG64(1501))
    qm = rng.standard_normal((2, 3, n_head, hd), dtype=np.float32)
    outm = pkg.decode_attention(torch.from_numpy(qm).cuda(), dev["k"], dev["v"], dev["positions"])
    torch.cuda.synchronize()
    refm = oracle.attn_decode_multi(qm, case["k"], case["v"], case["positions"], 3, n_head, n_kv,
                                    hd, cap, 1 / math.sqrt(hd), n_threads=8, kv_dtype=kv)
    assert_close(outm.cpu().numpy(), refm, "decode_attention %s, 3 rows" % kv)
    # each kernel by name
    for kernel in (pkg.ATTN_VARIANT_SIMT, pkg.ATTN_VARIANT_TC, pkg.ATTN_VARIANT_TCGEN05,
                   pkg.ATTN_VARIANT_TCGEN05_CLUSTER, pkg.ATTN_VARIANT_TC_TILE):
        outk = pkg.decode_attention(dev["q"], dev["k"], dev["v"], dev["positions"], kernel=kernel)
        torch.cuda.synchronize()
        assert_close(outk.cpu().numpy(), ref, "decode_attention %s kernel %d" % (kv, kernel))
