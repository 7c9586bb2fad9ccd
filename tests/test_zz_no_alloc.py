"""attn_decode_static -- the entry point for callers that cannot allocate
device memory at call time (a step under CUDA stream capture, a plugin whose
framework owns all device memory, a fixed memory budget). It keeps its scratch
in a fixed device array inside the library instead of a workspace.

Checked through the C ABI on two calls in a row (the array keeps the first
call's contents when the second one runs):
  - against the oracle, within the parity tolerance used everywhere else;
  - bit for bit against attn_decode_ex with its own workspace and the same
    arguments, n_splits = 0 included, for every kernel variant, the
    early-start flag and the bfloat16 cache: the split count the static call
    plans must be the one attn_decode_ex plans.
This file is collected last so that a failure here leaves every other test
already run.
"""
import ctypes
import math

import numpy as np
import pytest

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


def _oracle(host, n_head, n_kv, hd, cap, scale, kv_dtype):
    import oracle
    return oracle.attn_decode(host["q"], host["k"], host["v"], host["positions"], n_head, n_kv,
                              hd, cap, scale, n_threads=8, kv_dtype=kv_dtype)


def _ex_raw(pkg, dev, out, n_head, n_kv, hd, cap, scale, P, blk, variant):
    """attn_decode_ex with a workspace of exactly the size its own plan needs."""
    import torch
    lib = pkg.load()
    n_seq = dev["positions"].shape[0]
    if P:
        P_plan = P
    elif blk:
        P_plan = -(-cap // blk)                 # by block length: one split per block of rows
    else:
        P_plan = pkg.attn_split_heuristic_ex(n_seq, 1, n_head, n_kv, hd, cap, 0, variant)
    assert P_plan > 0
    ws = torch.empty(max(pkg.attn_workspace_size(n_seq, n_head, hd, P_plan), 256),
                     dtype=torch.uint8, device="cuda")
    st = lib.attn_decode_ex(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                            dev["positions"].data_ptr(), out.data_ptr(), n_seq, n_head, n_kv, hd,
                            ctypes.c_float(scale), cap, P, blk, variant, ws.data_ptr(),
                            ws.numel(), torch.cuda.current_stream().cuda_stream)
    return st, ws


def _static_raw(pkg, dev, out, n_head, n_kv, hd, cap, scale, P, blk, variant=0):
    import torch
    lib = pkg.load()
    return lib.attn_decode_static(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                                  dev["positions"].data_ptr(), out.data_ptr(),
                                  dev["positions"].shape[0], n_head, n_kv, hd, ctypes.c_float(scale),
                                  cap, P, blk, variant, torch.cuda.current_stream().cuda_stream)


CASES = [
    # (seed, n_head, n_kv, hd, cap, ctx per sequence, P, split_len)
    (31, 28, 4, 128, 4096, (4096,), 0, 0),
    (32, 16, 2, 256, 2000, (1999,), 0, 128),
    (33, 32, 8, 128, 1500, (1500, 7, 0, 999), 0, 0),
]


def _two_calls(pkg, case, variant, kv_dtype="f16"):
    """Two static calls in a row (different inputs, the second shorter), each
    against the oracle and bit for bit against attn_decode_ex."""
    import torch
    seed, n_head, n_kv, hd, cap, ctx, P, blk = case
    scale = 1 / math.sqrt(hd)
    first = make_case(seed, len(ctx), n_head, n_kv, hd, cap, ctx, kv_dtype=kv_dtype)
    second = make_case(seed + 100, len(ctx), n_head, n_kv, hd, cap,
                       tuple(max(c // 2, 1) for c in ctx), kv_dtype=kv_dtype)
    for host in (first, second):
        dev = to_device(host)
        out = torch.full_like(dev["q"], float("nan"))
        st = _static_raw(pkg, dev, out, n_head, n_kv, hd, cap, scale, P, blk, variant)
        if st == pkg.ATTN_ERR_UNSUPPORTED and (variant & 0xF) == pkg.ATTN_VARIANT_TCGEN05_CLUSTER:
            pytest.skip("this device cannot hold the fused kernel's 16-block cluster")
        assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
        ref_out = torch.full_like(dev["q"], float("nan"))
        st_ex, _ = _ex_raw(pkg, dev, ref_out, n_head, n_kv, hd, cap, scale, P, blk, variant)
        assert st_ex == pkg.ATTN_OK, pkg.attn_status_string(st_ex)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got, ref_out.cpu().numpy()), "static and ex differ (variant %#x)" % variant
        assert_close(got, _oracle(host, n_head, n_kv, hd, cap, scale, kv_dtype),
                     "static vs oracle (variant %#x)" % variant)


@pytest.mark.parametrize("case_idx", range(len(CASES)))
def test_static_scratch_matches_oracle_twice(pkg, case_idx):
    _two_calls(pkg, CASES[case_idx], 0)


@pytest.mark.parametrize("variant_name", ["TC", "TCGEN05", "TCGEN05_CLUSTER", "TC_TILE", "STABLE",
                                          "TCGEN05|STABLE", "TC_TILE|STABLE", "BF16"])
def test_static_scratch_every_variant_plans_like_ex(pkg, variant_name):
    """n_splits = 0 with an explicit kernel or flags: the static call must plan
    the split count attn_decode_ex plans for that variant (the cluster-fused
    kernel takes exactly 16 splits and no scratch; tcgen05 needs whole-tile
    splits; the early-start flag changes the count)."""
    names = {"TC": pkg.ATTN_VARIANT_TC, "TCGEN05": pkg.ATTN_VARIANT_TCGEN05,
             "TCGEN05_CLUSTER": pkg.ATTN_VARIANT_TCGEN05_CLUSTER, "STABLE": pkg.ATTN_KV_STABLE,
             "TCGEN05|STABLE": pkg.ATTN_VARIANT_TCGEN05 | pkg.ATTN_KV_STABLE,
             "TC_TILE": pkg.ATTN_VARIANT_TC_TILE,
             "TC_TILE|STABLE": pkg.ATTN_VARIANT_TC_TILE | pkg.ATTN_KV_STABLE,
             "BF16": pkg.ATTN_KV_BF16}
    variant = names[variant_name]
    _two_calls(pkg, CASES[0], variant, kv_dtype="bf16" if variant & pkg.ATTN_KV_BF16 else "f16")


def test_static_scratch_tcgen05_on_a_long_cache(pkg):
    """A capacity where variant 0 keeps the mma.sync kernel: the tcgen05 kernel
    needs P * 128 >= cap, which the static call's plan must honour."""
    _two_calls(pkg, (35, 28, 4, 128, 20000, (19999,), 0, 0), pkg.ATTN_VARIANT_TCGEN05)


def test_static_scratch_rejects_shapes_beyond_its_size(pkg):
    import torch
    n_head, n_kv, hd = 64, 8, 256
    dev = to_device(make_case(34, 1, n_head, n_kv, hd, 64, (64,)))
    out = torch.empty_like(dev["q"])
    P = 4000            # 64 heads x 4000 splits x 1 KB of partials: far past the fixed array
    assert pkg.attn_workspace_size(1, n_head, hd, P) > 8 * 1024 * 1024
    status = _static_raw(pkg, dev, out, n_head, n_kv, hd, 64, 1 / 16, P, 0)
    assert status == pkg.ATTN_ERR_WORKSPACE
