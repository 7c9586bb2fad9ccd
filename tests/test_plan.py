"""GPU: the planning entry points describe the call that variant 0 makes.

attn_resolve_variant and attn_split_heuristic_ex name a kernel and a split
count; a call with n_splits = 0 must then run exactly that plan. Each shape
below (the benchmark layers, two query rows, and both sides of the one-wave
boundary of the tcgen05 kernel) is run three ways: variant 0 with n_splits = 0
and a workspace of exactly attn_workspace_size(planned P) bytes; the resolved
variant forced with n_splits = P; and the oracle. The first two must agree bit
for bit (same kernel, same splits, same order of operations), and both must
match the oracle within the parity tolerance."""
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


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


# (n_seq, n_q, n_head, n_kv_head, head_dim, cap); the boundaries are the one-wave
# limits on a 152-SM device and are plain shapes elsewhere
SHAPES = [
    (1, 1, 28, 4, 128, 8192),          # the 7b layer
    (1, 1, 16, 2, 256, 8400),          # the long layer
    (1, 2, 28, 4, 128, 8192),          # two query rows: 14 slots per KV head
    (1, 4, 28, 4, 128, 2048),          # four rows: two query groups per KV head
    (1, 1, 28, 4, 128, 114 * 128),     # 456 one-tile blocks
    (1, 1, 28, 4, 128, 114 * 128 + 1),
    (2, 1, 28, 4, 128, 57 * 128 + 1),
    (1, 1, 16, 2, 256, 152 * 96 + 1),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("stable", [False, True])
def test_call_runs_the_planned_kernel_and_split_count(pkg, shape, stable):
    import torch
    n_seq, n_q, n_head, n_kv, hd, cap = shape
    flags = pkg.ATTN_KV_STABLE if stable else 0
    sms = _sms()
    P = pkg.attn_split_heuristic_ex(n_seq, n_q, n_head, n_kv, hd, cap, sms, flags)
    v = pkg.attn_resolve_variant(n_seq, n_q, n_head, n_kv, hd, cap, sms, flags)
    assert P > 0 and v in (pkg.ATTN_VARIANT_TC, pkg.ATTN_VARIANT_TCGEN05, pkg.ATTN_VARIANT_TC_TILE)
    ctx = tuple(cap - 3 - 17 * s for s in range(n_seq))
    case = make_case(7100 + cap % 97 + n_q, n_seq, n_head, n_kv, hd, cap, ctx)
    scale = 1 / math.sqrt(hd)
    if n_q > 1:
        rng = np.random.Generator(np.random.PCG64([cap, n_q]))
        case["q"] = rng.standard_normal((n_seq, n_q, n_head, hd), dtype=np.float32)
    dev = to_device(case)
    ws_bytes = pkg.attn_workspace_size(n_seq, n_q * n_head, hd, P)
    outs = []
    for variant, n_splits in ((flags, 0), (v | flags, P)):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.full_like(dev["q"], float("nan"))
        if n_q == 1:
            pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_head,
                               n_kv, hd, scale, cap, n_splits=n_splits, variant=variant,
                               workspace=ws, workspace_bytes=ws_bytes)
        else:
            pkg.attn_decode_multi(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_q,
                                  n_head, n_kv, hd, scale, cap, n_splits=n_splits, variant=variant,
                                  workspace=ws, workspace_bytes=ws_bytes)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    if n_q == 1:
        ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                                 hd, cap, scale, n_threads=8)
    else:
        ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                       n_head, n_kv, hd, cap, scale, n_threads=8)
    assert_close(outs[0], ref, "plan %s stable=%s: variant %d, P=%d" % (shape, stable, v, P))


@pytest.mark.parametrize("blk", [32, 64, 96, 128, 256])
def test_block_length_without_split_count_takes_one_split_per_block(pkg, blk):
    """By block length with n_splits = 0 the call takes P = ceil(cap / split_len)
    (Red Lite dev35 "Change": one split per block of positions): bit for bit the
    call with that P given, in a workspace of exactly that size; both match the
    oracle."""
    import torch
    n_head, n_kv, hd, cap = 16, 2, 256, 8400
    case = make_case(7300 + blk, 1, n_head, n_kv, hd, cap, (cap - 5,))
    dev = to_device(case)
    scale = 1 / math.sqrt(hd)
    P = -(-cap // blk)
    ws_bytes = pkg.attn_workspace_size(1, n_head, hd, P)
    outs = []
    for n_splits in (0, P):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.full_like(dev["q"], float("nan"))
        pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, 1, n_head, n_kv,
                           hd, scale, cap, n_splits=n_splits, split_len=blk, workspace=ws,
                           workspace_bytes=ws_bytes)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv, hd,
                             cap, scale, n_threads=8)
    assert_close(outs[0], ref, "block %d, n_splits 0 -> P %d" % (blk, P))


# (n_seq, n_q, n_head, n_kv_head, head_dim, cap, n_splits, split_len, variant flags)
PLAN_CALLS = [
    (1, 1, 28, 4, 128, 8192, 0, 0, 0),
    (1, 1, 28, 4, 128, 8192, 0, 0, 0x20),          # early start
    (1, 1, 16, 2, 256, 8400, 0, 32, 0),            # block 32: more blocks than one wave
    (1, 1, 16, 2, 256, 8400, 0, 64, 0),
    (1, 1, 16, 2, 256, 8400, 0, 128, 0),           # longer than a tcgen05 tile
    (1, 1, 28, 4, 128, 8192, 40, 0, 0),            # explicit count, fewer than 64 tiles
    (4, 1, 32, 8, 128, 3000, 0, 0, 0),
    (1, 4, 28, 4, 128, 2048, 0, 0, 0),
    (1, 2, 28, 4, 128, 8192, 0, 0, 0),
    (1, 1, 28, 4, 128, 4096, 0, 0, 4),             # cluster-fused: 16 splits, no workspace
]


@pytest.mark.parametrize("call", PLAN_CALLS, ids=lambda c: "x".join(map(str, c)))
def test_plan_call_is_the_call(pkg, call):
    """attn_plan_call names the kernel, split count and workspace of a call:
    the call in a workspace of exactly that size succeeds and equals, bit for
    bit, the same call with the named kernel and split count given."""
    import torch
    n_seq, n_q, n_head, n_kv, hd, cap, P_in, blk, flags = call
    try:
        v, P, ws_bytes = pkg.attn_plan_call(n_seq, n_q, n_head, n_kv, hd, cap, P_in, blk, flags)
    except pkg.AttnError as e:
        if (flags & 0xF) == pkg.ATTN_VARIANT_TCGEN05_CLUSTER and e.status == pkg.ATTN_ERR_UNSUPPORTED:
            pytest.skip("this device cannot hold the fused kernel's cluster")
        raise
    assert v in (pkg.ATTN_VARIANT_SIMT, pkg.ATTN_VARIANT_TC, pkg.ATTN_VARIANT_TCGEN05,
                 pkg.ATTN_VARIANT_TCGEN05_CLUSTER, pkg.ATTN_VARIANT_TC_TILE)
    want_ws = 0 if v == pkg.ATTN_VARIANT_TCGEN05_CLUSTER else pkg.attn_workspace_size(
        n_seq, n_q * n_head, hd, P)
    assert ws_bytes == want_ws
    if blk:
        assert P == (P_in or -(-cap // blk))
    ctx = tuple(cap - 1 - 13 * s for s in range(n_seq))
    case = make_case(7500 + cap % 89 + n_q, n_seq, n_head, n_kv, hd, cap, ctx)
    if n_q > 1:
        rng = np.random.Generator(np.random.PCG64([cap, n_q, 1]))
        case["q"] = rng.standard_normal((n_seq, n_q, n_head, hd), dtype=np.float32)
    dev = to_device(case)
    scale = 1 / math.sqrt(hd)
    outs = []
    for variant, n_splits in ((flags, P_in), ((flags & ~0xF) | v, P)):
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        out = torch.full_like(dev["q"], float("nan"))
        if n_q == 1:
            pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_head,
                               n_kv, hd, scale, cap, n_splits=n_splits, split_len=blk,
                               variant=variant, workspace=ws, workspace_bytes=ws_bytes)
        else:
            pkg.attn_decode_multi(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_q,
                                  n_head, n_kv, hd, scale, cap, n_splits=n_splits, split_len=blk,
                                  variant=variant, workspace=ws, workspace_bytes=ws_bytes)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    if n_q == 1:
        ref = oracle.attn_decode(case["q"], case["k"], case["v"], case["positions"], n_head, n_kv,
                                 hd, cap, scale, n_threads=8)
    else:
        ref = oracle.attn_decode_multi(case["q"], case["k"], case["v"], case["positions"], n_q,
                                       n_head, n_kv, hd, cap, scale, n_threads=8)
    assert_close(outs[0], ref, "plan %s: variant %d, P=%d" % (call, v, P))
