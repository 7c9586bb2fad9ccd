"""GPU parity for a bfloat16 KV cache (ATTN_KV_BF16): every compiled
(head_dim, group) pair on both kernels, split boundaries, NaN past nkv, the
fused append and a full-size workload, against the oracle's bfloat16 entry
points, at the same tolerance as the f16 cache (1e-4 + 1e-3 |ref|)."""
import math

import numpy as np
import pytest

import oracle
from decode_attention_gqa_gb300 import synthetic as syn
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


def _ref(case, n_head, n_kv, hd, cap, scale):
    return oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                              hd, cap, scale, n_threads=8, kv_dtype="bf16")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("hd", [8, 64, 128, 256])
def test_bf16_all_groups_and_head_dims(pkg, hd, variant):
    if variant == 2 and hd % 16:
        pytest.skip("the tensor-core kernel needs head_dim % 16 == 0")
    for G in (1, 2, 4, 7, 8):
        n_kv, cap = 2, 700
        n_head = G * n_kv
        case = make_case(300 * hd + G, 1, n_head, n_kv, hd, cap, (613,), kv_dtype="bf16")
        scale = 1 / math.sqrt(hd)
        got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale, n_splits=5,
                         variant=variant | pkg.ATTN_KV_BF16).cpu().numpy()
        assert_close(got, _ref(case, n_head, n_kv, hd, cap, scale), "bf16 hd%d G%d" % (hd, G))


@pytest.mark.parametrize("variant", [1, 2])
def test_bf16_boundaries_and_nan_tail(pkg, variant):
    n_head, n_kv, hd, cap = 32, 8, 128, 900
    ctx = (1, 900, 0, 17, 450, 899, 64, 333)
    case = make_case(301, len(ctx), n_head, n_kv, hd, cap, ctx, k_scale=4.0, fill=np.nan,
                     kv_dtype="bf16")
    scale = 1 / math.sqrt(hd)
    ref = _ref(case, n_head, n_kv, hd, cap, scale)
    for P, blk in ((0, 0), (4, 0), (15, 64)):
        got = run_decode(pkg, to_device(case), n_head, n_kv, hd, cap, scale, n_splits=P,
                         split_len=blk, variant=variant | pkg.ATTN_KV_BF16).cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_close(got, ref, "bf16 ragged P=%d blk=%d" % (P, blk))


@pytest.mark.parametrize("variant", [1, 2])
def test_bf16_append(pkg, variant):
    import torch
    n_head, n_kv, hd, cap = 16, 2, 256, 400
    nkv = 333
    case = make_case(302, 1, n_head, n_kv, hd, cap, (nkv,), kv_dtype="bf16")
    rng = np.random.Generator(np.random.PCG64(303))
    k_new = syn.to_bf16_bits(rng.standard_normal((1, n_kv, hd), dtype=np.float32))
    v_new = syn.to_bf16_bits(rng.standard_normal((1, n_kv, hd), dtype=np.float32))
    case["k"][0, nkv - 1] = 0x7FC0                         # stale NaN where the new row goes
    case["v"][0, nkv - 1] = 0x7FC0
    dev = to_device(case)
    kn = torch.from_numpy(k_new.view(np.int16)).cuda()
    vn = torch.from_numpy(v_new.view(np.int16)).cuda()
    out = torch.full_like(dev["q"], float("nan"))
    pkg.attn_decode_append(dev["q"], kn, vn, dev["k"], dev["v"], dev["positions"], out, 1, n_head,
                           n_kv, hd, 1 / 16, cap, variant=variant | pkg.ATTN_KV_BF16)
    torch.cuda.synchronize()
    kh, vh = case["k"].copy(), case["v"].copy()
    kh[0, nkv - 1], vh[0, nkv - 1] = k_new[0], v_new[0]
    ref = oracle.attn_decode(case["q"], kh, vh, case["positions"], n_head, n_kv, hd, cap, 1 / 16,
                             kv_dtype="bf16")
    assert_close(out.cpu().numpy(), ref, "bf16 append")
    np.testing.assert_array_equal(dev["k"].cpu().numpy().view(np.uint16), kh)


def test_bf16_full_7b_workload(pkg):
    w = syn.WORKLOADS["7b"]
    lay = syn.make_layer(w, kv_dtype="bf16")
    got = run_decode(pkg, to_device(lay), w.n_head, w.n_kv_head, w.head_dim, w.cap, w.scale,
                     variant=pkg.ATTN_KV_BF16).cpu().numpy()
    ref = oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                             w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=16,
                             kv_dtype="bf16")
    assert_close(got, ref, "bf16 7b")


def test_bf16_static_entry_point(pkg):
    import torch
    n_head, n_kv, hd, cap = 8, 2, 128, 600
    case = make_case(304, 1, n_head, n_kv, hd, cap, (555,), kv_dtype="bf16")
    dev = to_device(case)
    out = torch.full_like(dev["q"], float("nan"))
    pkg.attn_decode_static(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv,
                           hd, 1 / math.sqrt(hd), cap, variant=pkg.ATTN_KV_BF16)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), _ref(case, n_head, n_kv, hd, cap, 1 / math.sqrt(hd)),
                 "bf16 static")
