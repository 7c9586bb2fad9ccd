"""attn_decode_static -- the entry point for callers that cannot allocate
device memory at call time (a step under CUDA stream capture, a plugin whose
framework owns all device memory, a fixed memory budget). It keeps its scratch
in a fixed device array inside the library instead of a workspace.

Checked through the C ABI against attn_decode_ex with a caller workspace, on
two calls in a row (the array keeps the first call's contents when the second
one runs), within the parity tolerance used everywhere else. This file is
collected last so that a failure here leaves every other test already run.
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


def _reference(pkg, dev, n_head, n_kv, hd, cap, scale, P, blk):
    import torch
    out = torch.full_like(dev["q"], float("nan"))
    n_seq = dev["positions"].shape[0]
    P_ref = P or pkg.attn_split_heuristic(n_seq, n_head, n_kv, hd, cap, 0)
    ws = torch.empty(pkg.attn_workspace_size(n_seq, n_head, hd, P_ref), dtype=torch.uint8,
                     device="cuda")
    pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_head, n_kv,
                       hd, scale, cap, n_splits=P_ref, split_len=blk, workspace=ws)
    return out


def _static_raw(pkg, dev, out, n_head, n_kv, hd, cap, scale, P, blk):
    import torch
    lib = pkg.load()
    return lib.attn_decode_static(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                                  dev["positions"].data_ptr(), out.data_ptr(),
                                  dev["positions"].shape[0], n_head, n_kv, hd, ctypes.c_float(scale),
                                  cap, P, blk, 0, torch.cuda.current_stream().cuda_stream)


CASES = [
    # (seed, n_head, n_kv, hd, cap, ctx per sequence, P, split_len)
    (31, 28, 4, 128, 4096, (4096,), 0, 0),
    (32, 16, 2, 256, 2000, (1999,), 0, 128),
    (33, 32, 8, 128, 1500, (1500, 7, 0, 999), 0, 0),
]


@pytest.mark.parametrize("case_idx", range(len(CASES)))
def test_static_scratch_matches_workspace_path_twice(pkg, case_idx):
    import torch
    seed, n_head, n_kv, hd, cap, ctx, P, blk = CASES[case_idx]
    scale = 1 / math.sqrt(hd)
    first = to_device(make_case(seed, len(ctx), n_head, n_kv, hd, cap, ctx))
    second = to_device(make_case(seed + 100, len(ctx), n_head, n_kv, hd, cap,
                                 tuple(max(c // 2, 1) for c in ctx)))
    for dev in (first, second):              # two calls in a row share the array
        out = torch.full_like(dev["q"], float("nan"))
        assert _static_raw(pkg, dev, out, n_head, n_kv, hd, cap, scale, P, blk) == pkg.ATTN_OK
        ref = _reference(pkg, dev, n_head, n_kv, hd, cap, scale, P, blk)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), "static vs ex")


def test_static_scratch_rejects_shapes_beyond_its_size(pkg):
    import torch
    n_head, n_kv, hd, cap = 64, 8, 256, 4096
    dev = to_device(make_case(34, 1, n_head, n_kv, hd, 64, (64,)))
    out = torch.empty_like(dev["q"])
    P = 4000            # 64 heads x 4000 splits x 1 KB of partials: far past the fixed array
    assert pkg.attn_workspace_size(1, n_head, hd, P) > 8 * 1024 * 1024
    status = _static_raw(pkg, dev, out, n_head, n_kv, hd, 64, 1 / 16, P, 0)
    assert status == pkg.ATTN_ERR_WORKSPACE
