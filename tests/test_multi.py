"""GPU: several causal query rows per sequence (attn_decode_multi) against the
oracle's multi-query definition: query row t of a sequence with nkv rows sits
at position nkv - n_q + t and attends rows [0, nkv - n_q + t] (dotLLM #199 §2:
the causal mask's offset is the query's position)."""
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


def _case(seed, n_seq, n_q, n_head, n_kv, hd, cap, ctx, kv_dtype="f16", k_scale=1.0, fill=0.0):
    c = make_case(seed, n_seq, n_head, n_kv, hd, cap, ctx, kv_dtype=kv_dtype, k_scale=k_scale,
                  fill=fill)
    rng = np.random.Generator(np.random.PCG64([seed, 9]))
    c["q"] = rng.standard_normal((n_seq, n_q, n_head, hd), dtype=np.float32)
    return c


def _run(pkg, case, n_q, n_head, n_kv, hd, cap, scale, P=0, blk=0, variant=0):
    import torch
    dev = to_device(case)
    out = torch.full_like(dev["q"], float("nan"))
    n_seq = case["positions"].shape[0]
    pkg.attn_decode_multi(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_q, n_head,
                          n_kv, hd, scale, cap, n_splits=P, split_len=blk, variant=variant)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# 2 forces the mma.sync streaming multi-query kernel, 3 the tcgen05 kernel and 5 the
# one-tile mma.sync kernel (16 slots per block each); variant 0 takes the one-tile kernel
# at head_dim 128 where its blocks fit one wave, else tcgen05 where a KV head's n_q x G
# slots fit one block, else the streaming kernel
@pytest.mark.parametrize("variant", [0, 2, 3, 5])
@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("kv", ["f16", "bf16"])
def test_multi_query_shapes(pkg, hd, kv, variant):
    if variant == 3 and hd == 64:
        pytest.skip("the tcgen05 kernel is built for head_dim 128 and 256")
    if variant == 5 and hd != 128:
        pytest.skip("the one-tile kernel takes several query rows at head_dim 128")
    flag = (pkg.ATTN_KV_BF16 if kv == "bf16" else 0) | variant
    for (G, n_q) in ((1, 2), (4, 3), (7, 2), (8, 2), (7, 4), (2, 9)):
        n_kv, cap = 2, 500
        n_head = G * n_kv
        case = _case(hd * 10 + G * 3 + n_q, 1, n_q, n_head, n_kv, hd, cap, (437,), kv)
        scale = 1 / math.sqrt(hd)
        got = _run(pkg, case, n_q, n_head, n_kv, hd, cap, scale, variant=flag)
        ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                       n_head, n_kv, hd, cap, scale, n_threads=8, kv_dtype=kv)
        assert_close(got, ref, "multi hd%d G%d n_q%d %s variant %d" % (hd, G, n_q, kv, variant))


@pytest.mark.parametrize("variant", [0, 3, 5])
def test_multi_query_short_contexts_and_boundaries(pkg, variant):
    n_q, n_head, n_kv, hd, cap = 4, 28, 4, 128, 1024
    scale = 1 / math.sqrt(hd)
    splits = ((0, 0), (7, 0), (17, 64)) if variant == 0 else ((0, 0), (8, 0), (17, 64), (9, 128))   # tile 128
    for nkv in (1, 2, 3, 4, 5, 16, 17, 63, 64, 65, 112, 113, 127, 128, 129, 1000, 1024):
        case = _case(500 + nkv, 1, n_q, n_head, n_kv, hd, cap, (nkv,))
        for P, blk in splits:
            got = _run(pkg, case, n_q, n_head, n_kv, hd, cap, scale, P, blk, variant)
            ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                           n_head, n_kv, hd, cap, scale, n_threads=8)
            assert_close(got, ref, "multi nkv=%d P=%d blk=%d" % (nkv, P, blk))
            if nkv < n_q:                         # queries before the first cached row
                assert np.all(got[0, :n_q - nkv] == 0)


@pytest.mark.parametrize("variant", [0, 3, 5])
def test_multi_query_ragged_batch_and_large_spread(pkg, variant):
    n_q, n_head, n_kv, hd, cap = 3, 32, 8, 128, 900
    ctx = (2, 900, 0, 17, 450, 899, 64, 333)
    case = _case(600, len(ctx), n_q, n_head, n_kv, hd, cap, ctx, k_scale=6.0, fill=np.nan)
    scale = 1 / math.sqrt(hd)
    got = _run(pkg, case, n_q, n_head, n_kv, hd, cap, scale, variant=variant)
    ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                   n_head, n_kv, hd, cap, scale, n_threads=8)
    assert_close(got, ref, "multi ragged")
    assert np.all(np.isfinite(got))


def test_multi_query_one_row_matches_single_query(pkg):
    import torch
    n_head, n_kv, hd, cap = 16, 2, 256, 700
    case = _case(700, 1, 1, n_head, n_kv, hd, cap, (650,))
    got = _run(pkg, case, 1, n_head, n_kv, hd, cap, 0.0625)
    single = dict(case, q=case["q"][:, 0])
    ref = oracle.attn_decode(single["q"], single["k"], single["v"], single["positions"], n_head,
                             n_kv, hd, cap, 0.0625)
    assert_close(got[:, 0], ref, "n_q = 1")


def test_multi_query_rejections(pkg):
    import torch
    q = torch.zeros(1, 2, 4, 8, device="cuda")
    kv = torch.zeros(1, 16, 2, 8, dtype=torch.float16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = pkg.load()
    st = lib.attn_decode_multi(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), pos.data_ptr(),
                               q.data_ptr(), 1, 2, 4, 2, 8, 1.0, 16, 0, 0, 0, None, 0, None)
    assert st == pkg.ATTN_ERR_UNSUPPORTED                     # head_dim 8: tensor cores only
    q2 = torch.zeros(1, 2, 4, 128, device="cuda")
    kv2 = torch.zeros(1, 16, 2, 128, dtype=torch.float16, device="cuda")
    st = lib.attn_decode_multi(q2.data_ptr(), kv2.data_ptr(), kv2.data_ptr(), pos.data_ptr(),
                               q2.data_ptr(), 1, 2, 4, 2, 128, 1.0, 16, 0, 0, pkg.ATTN_VARIANT_SIMT,
                               None, 0, None)
    assert st == pkg.ATTN_ERR_UNSUPPORTED
    q3 = torch.zeros(1, 2, 4, 256, device="cuda")
    kv3 = torch.zeros(1, 16, 2, 256, dtype=torch.float16, device="cuda")
    st = lib.attn_decode_multi(q3.data_ptr(), kv3.data_ptr(), kv3.data_ptr(), pos.data_ptr(),
                               q3.data_ptr(), 1, 2, 4, 2, 256, 1.0, 16, 0, 0, pkg.ATTN_VARIANT_TC_TILE,
                               None, 0, None)
    assert st == pkg.ATTN_ERR_UNSUPPORTED                     # one-tile kernel, several rows: hd 128
    st = lib.attn_decode_multi(q2.data_ptr(), kv2.data_ptr(), kv2.data_ptr(), pos.data_ptr(),
                               q2.data_ptr(), 1, 0, 4, 2, 128, 1.0, 16, 0, 0, 0, None, 0, None)
    assert st == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("variant", [0, 3, 5])
@pytest.mark.parametrize("n_q, G, nkv", [(64, 4, 300), (50, 8, 20), (33, 1, 700), (128, 7, 1000)])
def test_many_query_rows(pkg, n_q, G, nkv, variant):
    """Prefill-sized chunks: many query groups per KV head (up to 56 blocks
    along y), and with n_q > nkv the first n_q - nkv rows see no cache row."""
    n_kv, hd, cap = 2, 128, 1024
    n_head = G * n_kv
    case = _case(800 + n_q + G, 1, n_q, n_head, n_kv, hd, cap, (nkv,))
    got = _run(pkg, case, n_q, n_head, n_kv, hd, cap, 1 / math.sqrt(hd), variant=variant)
    ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q, n_head,
                                   n_kv, hd, cap, 1 / math.sqrt(hd), n_threads=8)
    assert_close(got, ref, "n_q=%d G=%d nkv=%d variant %d" % (n_q, G, nkv, variant))
    if n_q > nkv:
        assert np.all(got[0, :n_q - nkv] == 0)
