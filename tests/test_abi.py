"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/*.h, and its host-only logic (argument validation, split
heuristic, workspace sizing, status strings) behaves as documented. Nothing
here launches a kernel."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import decode_attention_gqa_gb300 as pkg
from decode_attention_gqa_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return pkg.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("attn_decode", "attn_decode_ex", "attn_split_heuristic", "attn_workspace_size",
                 "attn_read_device_error", "attn_status_string"):
        assert want in names


def test_binding_constants_match_the_header():
    """Every ATTN_* macro and enumerator of the header has the same value in the binding."""
    text = open(os.path.join(ROOT, "include", "attn_decode.h")).read()
    found = 0
    for m in re.finditer(r"^#define (ATTN_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text, flags=re.M):
        name, val = m.group(1), int(m.group(2), 0)
        if name in ("ATTN_STATIC_SCRATCH_BYTES",) or not hasattr(pkg, name):
            continue
        assert getattr(pkg, name) == val, name
        found += 1
    for m in re.finditer(r"^\s*(ATTN_(?:OK|ERR_\w+))\s*=\s*(\d+)", text, flags=re.M):
        assert getattr(pkg, m.group(1)) == int(m.group(2)), m.group(1)
        found += 1
    assert found >= 12
    assert pkg.ATTN_KV_STABLE & pkg.ATTN_KV_BF16 == 0


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(pkg.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), "missing export %s" % name


def test_version_and_status_strings(lib):
    assert pkg.attn_version() == 10000
    assert pkg.attn_status_string(pkg.ATTN_OK) == "ATTN_OK"
    assert pkg.attn_status_string(pkg.ATTN_ERR_WORKSPACE) == "ATTN_ERR_WORKSPACE"
    assert pkg.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


def test_workspace_size(lib):
    # partial accumulators [n_seq][n_head][P][hd] f32 + (mx, S) pairs, each 256-aligned
    assert pkg.attn_workspace_size(1, 28, 128, 38) == 28 * 38 * 128 * 4 + ((28 * 38 * 8 + 255) // 256 * 256)
    assert pkg.attn_workspace_size(0, 28, 128, 38) == 0
    assert pkg.attn_workspace_size(1, 28, 128, 0) == 0


def test_split_heuristic_host_only(lib):
    # an explicit SM count never touches the device
    P = pkg.attn_split_heuristic(1, 28, 4, 128, 8192, 152)
    assert 1 <= P <= 8192 // 16
    # more independent (sequence, KV head) units -> fewer splits each
    assert pkg.attn_split_heuristic(32, 32, 8, 128, 32768, 152) <= P
    # a short head_dim-128 call runs the tcgen05 kernel, one 128-row tile per split:
    # 40 rows -> 1 split; the mma.sync kernel's splits are whole 64-row tiles: also 1;
    # the cluster-fused form always takes 16 splits
    assert pkg.attn_split_heuristic(1, 8, 2, 128, 40, 152) == 1
    assert pkg.attn_split_heuristic_ex(1, 1, 8, 2, 128, 40, 152, pkg.ATTN_VARIANT_TC) == 1
    assert pkg.attn_split_heuristic_ex(1, 1, 8, 2, 128, 8192, 152,
                                       pkg.ATTN_VARIANT_TCGEN05_CLUSTER) == 16
    # ... and the CUDA-core kernel's are 32-row warp slices: 40 rows -> 2 splits
    assert pkg.attn_split_heuristic_ex(1, 1, 8, 2, 128, 40, 152, pkg.ATTN_VARIANT_SIMT) == 2
    # one sequence, 28/4 heads at 8192 rows: variant 0 is the one-tile kernel with its
    # 256-row tiles, one block per SM: 152 / 4 = 38 splits of 216 -> 224 rows (more than
    # three quarters of the tile); the mma.sync kernel fills one wave, 4 x 64 blocks of
    # 128 rows; at 148 SMs 37 splits of 222 -> 224 rows; at 6000 rows one block per SM
    # would make 158-row chunks, so 128-row tiles, ceil(6000 / 128) = 47
    assert pkg.attn_split_heuristic(1, 28, 4, 128, 8192, 152) == 38
    assert pkg.attn_split_heuristic_ex(1, 1, 28, 4, 128, 8192, 152, pkg.ATTN_VARIANT_TC) == 64
    assert pkg.attn_split_heuristic(1, 28, 4, 128, 8192, 148) == 37
    assert pkg.attn_split_heuristic(1, 28, 4, 128, 6000, 152) == 47
    # a batch aims at eight waves so ragged lengths still balance
    assert pkg.attn_split_heuristic(32, 32, 8, 128, 32768, 152) == 10
    # unknown capacity: one wave of blocks over the (sequence, KV head) units
    assert pkg.attn_split_heuristic(1, 28, 4, 128, 0, 152) >= 152 // 4
    # rejected shapes
    assert pkg.attn_split_heuristic(1, 28, 5, 128, 8192, 152) == 0
    assert pkg.attn_split_heuristic(1, 18, 2, 128, 8192, 152) == 0      # group 9
    assert pkg.attn_split_heuristic(1, 8, 2, 96, 8192, 152) == 0        # head_dim 96


def test_split_heuristic_for_flagged_calls(lib):
    def h(n_seq, n_head, n_kv, hd, cap, sms, variant, n_q=1):
        return pkg.attn_split_heuristic_ex(n_seq, n_q, n_head, n_kv, hd, cap, sms, variant)
    # the plain call and variant 0 agree; the element type does not change P
    assert h(1, 28, 4, 128, 8192, 152, 0) == pkg.attn_split_heuristic(1, 28, 4, 128, 8192, 152)
    assert h(1, 28, 4, 128, 8192, 152, pkg.ATTN_KV_BF16) == 38
    # variant 0 on this short call is the one-tile kernel (256-row tiles, 38 balanced
    # splits); tcgen05 takes one 128-row tile per split
    S, TC, T5 = pkg.ATTN_KV_STABLE, pkg.ATTN_VARIANT_TC, pkg.ATTN_VARIANT_TCGEN05
    assert h(1, 28, 4, 128, 8192, 152, S) == 38 and h(1, 28, 4, 128, 8192, 152, T5 | S) == 64
    assert h(1, 28, 4, 128, 8192, 152, S | pkg.ATTN_KV_BF16) == 38
    assert h(1, 28, 4, 128, 2048, 152, S) == 16
    # mma.sync kernel, early start, one sequence: one block per SM would give each
    # block 256 rows, more than its 3 x 64-row stage ring, so blocks of 192 rows: 4 x 43
    assert h(1, 28, 4, 128, 8192, 152, TC | S) == 43
    assert h(1, 28, 4, 128, 8192, 152, TC | S | pkg.ATTN_KV_BF16) == 43
    # a shorter cache fits the ring at one block per SM: 2048 x 4 / 152 -> 64 rows
    assert h(1, 28, 4, 128, 2048, 152, TC | S) == 32
    # a long call keeps every resident block: 131072 rows x 8 KV heads
    assert h(1, 64, 8, 128, 131072, 152, pkg.ATTN_KV_STABLE) == h(1, 64, 8, 128, 131072, 152, 0) == 38
    # a batch keeps its eight waves
    assert h(32, 32, 8, 128, 32768, 152, pkg.ATTN_KV_STABLE) == 10
    # head_dim 256: variant 0 runs the one-tile kernel; the mma.sync kernel already runs
    # one block per SM
    assert h(1, 16, 2, 256, 8400, 152, S) == h(1, 16, 2, 256, 8400, 152, 0) == 76
    # ... with 128-row tiles, one block per SM: 152 / 2 = 76 splits of 111 -> 112 rows; at
    # 148 SMs 74 splits of 114 -> 128; a shorter cache keeps the 96-row tiles
    assert h(1, 16, 2, 256, 8400, 148, 0) == 74
    assert h(1, 16, 2, 256, 6000, 152, 0) == 63
    assert h(1, 16, 2, 256, 2048, 152, 0) == 22
    assert h(1, 16, 2, 256, 8400, 152, TC | S) == h(1, 16, 2, 256, 8400, 152, TC) == 75
    # several query rows: 4 rows x 7 heads = 28 pairs -> 2 query groups of 16 per KV
    # head; at one block per SM a block would hold 431 rows (not a short call), so
    # two blocks per SM: 8 x 37 blocks of 224 rows
    assert h(1, 28, 4, 128, 8192, 152, pkg.ATTN_KV_STABLE, n_q=4) == 37
    # short: one 128-row tile per split on the one-tile kernel, 16 x 4 x 2 blocks
    assert h(1, 28, 4, 128, 2048, 152, pkg.ATTN_KV_STABLE, n_q=4) == 16
    # 2 rows x 7 heads = 14 pairs: one group, so variant 0 runs the one-tile kernel with its
    # 256-row tiles, 38 balanced splits; the streaming mma.sync kernel keeps its ring-sized
    # blocks
    assert h(1, 28, 4, 128, 8192, 152, pkg.ATTN_KV_STABLE, n_q=2) == 38
    assert h(1, 28, 4, 128, 8192, 152, TC | S, n_q=2) == 43
    assert h(1, 28, 4, 128, 8192, 152, pkg.ATTN_VARIANT_SIMT, n_q=2) == 0  # tensor cores only
    # the CUDA-core kernel has its own granule and residency
    assert h(1, 28, 4, 128, 8192, 152, pkg.ATTN_VARIANT_SIMT) >= 1
    assert h(1, 28, 4, 128, 8192, 152, 7) == 0                           # no such variant
    assert h(1, 28, 4, 128, 8192, 152, 0, n_q=0) == 0


def test_resolved_variant(lib):
    r = pkg.attn_resolve_variant
    S, B = pkg.ATTN_KV_STABLE, pkg.ATTN_KV_BF16
    T5, TC, SI = pkg.ATTN_VARIANT_TCGEN05, pkg.ATTN_VARIANT_TC, pkg.ATTN_VARIANT_SIMT
    VT = pkg.ATTN_VARIANT_TC_TILE
    # variant 0: the one-tile mma.sync kernel for a short call (several query rows at
    # head_dim 128); the tcgen05 kernel for several query rows at head_dim 256
    assert r(1, 1, 28, 4, 128, 8192, 152, 0) == VT
    assert r(1, 1, 28, 4, 128, 8192, 152, S | B) == VT
    assert r(1, 1, 8, 2, 128, 40, 152, 0) == VT
    # the cluster-fused form only on request
    assert r(1, 1, 28, 4, 128, 2048, 152, pkg.ATTN_VARIANT_TCGEN05_CLUSTER) == \
        pkg.ATTN_VARIANT_TCGEN05_CLUSTER
    assert r(1, 1, 16, 2, 256, 2048, 152, pkg.ATTN_VARIANT_TCGEN05_CLUSTER) == 0
    assert r(1, 1, 16, 2, 256, 8400, 152, 0) == VT
    # ... the mma.sync kernel for long caches, batches, several query rows, head_dim
    # 64 and an unknown capacity; CUDA cores for head_dim 8
    assert r(1, 1, 64, 8, 128, 131072, 152, 0) == TC
    assert r(32, 1, 32, 8, 128, 32768, 152, 0) == TC
    assert r(1, 4, 28, 4, 128, 8192, 152, 0) == TC                 # 2 x 4 x 64 blocks > 3 x 152
    assert r(1, 2, 28, 4, 128, 8192, 152, 0) == VT                 # 14 slots: one group
    assert r(1, 2, 28, 4, 128, 8192, 152, S) == VT
    assert r(1, 3, 28, 4, 128, 8192, 152, 0) == TC                 # 21 slots
    assert r(1, 4, 28, 4, 128, 2048, 152, 0) == VT                 # 2 x 4 x 16 blocks
    assert r(1, 2, 28, 4, 128, 57 * 128, 152, 0) == VT             # 4 x 114 blocks, 3 per SM
    assert r(1, 2, 28, 4, 128, 114 * 128 + 1, 152, 0) == TC        # a second wave
    # 16 slots at head_dim 256: one block per SM, so 2 x 88 blocks are a second wave
    assert r(1, 2, 16, 2, 256, 8400, 152, 0) == TC
    assert r(1, 2, 16, 2, 256, 76 * 96, 152, 0) == T5
    assert r(1, 1, 8, 2, 64, 1024, 152, 0) == TC
    assert r(1, 1, 28, 4, 128, 0, 152, 0) == TC
    assert r(1, 1, 4, 2, 8, 64, 152, 0) == SI
    # the boundary: one wave of one-tile blocks, 3 per SM at head_dim 128 (4 x 114 = 456
    # blocks of 128 rows), 2 at head_dim 256 (2 x 152 = 304 blocks of 96 rows)
    assert r(1, 1, 28, 4, 128, 114 * 128, 152, 0) == VT
    assert r(1, 1, 28, 4, 128, 114 * 128 + 1, 152, 0) == TC
    assert r(1, 1, 28, 4, 128, 114 * 128 + 1, 152, S) == TC
    assert r(1, 1, 16, 2, 256, 152 * 96, 152, 0) == VT
    assert r(1, 1, 16, 2, 256, 152 * 96 + 1, 152, 0) == TC
    assert r(2, 1, 28, 4, 128, 57 * 128, 152, 0) == VT            # 2 sequences x 4 x 57
    assert r(2, 1, 28, 4, 128, 57 * 128 + 1, 152, 0) == TC
    # explicit variants are kept; tcgen05 is built for head_dim 128 and one query row
    assert r(1, 1, 28, 4, 128, 8192, 152, SI) == SI
    assert r(1, 1, 28, 4, 128, 8192, 152, TC) == TC
    assert r(1, 1, 64, 8, 128, 131072, 152, T5) == T5
    assert r(1, 1, 8, 2, 64, 1024, 152, T5) == 0
    assert r(1, 2, 8, 2, 128, 1024, 152, T5) == T5                         # several query rows too
    assert r(1, 1, 28, 4, 256, 8192, 152, VT) == VT                        # explicit one-tile kernel
    assert r(1, 2, 8, 2, 128, 1024, 152, VT) == VT                         # several rows: hd 128
    assert r(1, 2, 8, 2, 256, 1024, 152, VT) == 0
    assert r(1, 1, 8, 2, 64, 1024, 152, VT) == 0
    assert r(1, 1, 28, 5, 128, 8192, 152, 0) == 0


def _ex(lib, **kw):
    a = dict(q=16, k=16, v=16, pos=16, out=16, n_seq=1, n_head=8, n_kv=2, hd=128, scale=0.1,
             cap=64, P=0, blk=0, variant=0, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.attn_decode_ex(a["q"], a["k"], a["v"], a["pos"], a["out"], a["n_seq"], a["n_head"],
                              a["n_kv"], a["hd"], a["scale"], a["cap"], a["P"], a["blk"],
                              a["variant"], a["ws"], a["ws_bytes"], None)


def test_argument_validation_is_synchronous(lib):
    # Every case below is rejected on the host before any CUDA call.
    assert _ex(lib, n_head=8, n_kv=3) == pkg.ATTN_ERR_INVALID_ARG          # 8 % 3 != 0
    assert _ex(lib, n_kv=0) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, q=None) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, k=8) == pkg.ATTN_ERR_INVALID_ARG                        # misaligned
    assert _ex(lib, out=4) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, cap=0) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, P=-1) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, P=5000) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, blk=-3) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, variant=7) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, scale=float("nan")) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, scale=float("inf")) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, n_seq=-1) == pkg.ATTN_ERR_INVALID_ARG
    assert _ex(lib, ws=16) == pkg.ATTN_ERR_INVALID_ARG                      # not 256-aligned
    assert _ex(lib, n_seq=2, cap=2 ** 30) == pkg.ATTN_ERR_INVALID_ARG       # rows past int32
    assert _ex(lib, hd=96) == pkg.ATTN_ERR_UNSUPPORTED
    assert _ex(lib, hd=32) == pkg.ATTN_ERR_UNSUPPORTED
    assert _ex(lib, n_head=18, n_kv=2) == pkg.ATTN_ERR_UNSUPPORTED          # group 9
    # nothing to do: no launch, no CUDA call
    assert _ex(lib, n_seq=0, q=None, k=None, v=None, pos=None, out=None) == pkg.ATTN_OK
    # the single-sequence entry point
    assert lib.attn_decode(16, 16, 16, 16, 16, 2, 8, 2, 128, 0.1, None) == pkg.ATTN_ERR_INVALID_ARG


def test_plan_call_checks_its_arguments_before_the_device(lib):
    """attn_plan_call answers every shape error the call would answer, before it
    asks for the device (so here, without one, they still come back as such)."""
    import ctypes
    v, p, ws = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_size_t(7)

    def plan(n_seq=1, n_q=1, n_head=8, n_kv=2, hd=128, cap=64, P=0, blk=0, variant=0):
        return lib.attn_plan_call(n_seq, n_q, n_head, n_kv, hd, cap, P, blk, variant,
                                  ctypes.byref(v), ctypes.byref(p), ctypes.byref(ws))
    assert plan(n_head=8, n_kv=3) == pkg.ATTN_ERR_INVALID_ARG
    assert plan(cap=0) == pkg.ATTN_ERR_INVALID_ARG
    assert plan(P=5000) == pkg.ATTN_ERR_INVALID_ARG
    assert plan(variant=7) == pkg.ATTN_ERR_INVALID_ARG
    assert plan(n_q=0) == pkg.ATTN_ERR_INVALID_ARG
    assert plan(n_seq=0) == pkg.ATTN_ERR_INVALID_ARG        # nothing to plan
    assert plan(hd=96) == pkg.ATTN_ERR_UNSUPPORTED
    assert plan(n_head=18, n_kv=2) == pkg.ATTN_ERR_UNSUPPORTED
    assert plan(n_q=2, hd=8) == pkg.ATTN_ERR_UNSUPPORTED
    assert (v.value, p.value, ws.value) == (-1, -1, 7)       # outputs untouched on error


def test_binding_raises_attn_error(lib):
    with pytest.raises(pkg.AttnError) as ei:
        pkg.attn_decode_ex(16, 16, 16, 16, 16, 1, 8, 3, 128, 0.1, 64, stream=0)
    assert ei.value.status == pkg.ATTN_ERR_INVALID_ARG


def test_ptxas_reports_no_spills(lib):
    rep = cuda_build.spill_report()
    assert rep, "no ptxas report found"
    for fn, r in rep.items():
        assert r["spill_stores"] == 0 and r["spill_loads"] == 0 and r["stack"] == 0, fn


def test_selftest_limit_is_checked_before_any_launch(lib):
    # the bounded-wait self-test takes 1 ns .. 1 s, like the kernels' own waits
    assert lib.attn_selftest_bounded_wait(0, None) == pkg.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_bounded_wait(2_000_000_000, None) == pkg.ATTN_ERR_INVALID_ARG


def test_plain_c99_program_links_and_calls_the_host_entry_points(lib, tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links the
    library and calls the host-only entry points (no GPU needed)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_abi.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "attn_decode.h"
int main(void) {
    if (attn_version() <= 0) return 1;
    if (strcmp(attn_status_string(ATTN_ERR_WORKSPACE), "ATTN_ERR_WORKSPACE") != 0) return 2;
    if (attn_workspace_size(1, 28, 128, 37) == 0) return 3;
    if (attn_split_heuristic(1, 28, 4, 128, 8192, 152) != 38) return 4;
    if (attn_split_heuristic_ex(1, 1, 28, 4, 128, 8192, 152, ATTN_KV_STABLE | ATTN_VARIANT_TC) != 43)
        return 5;
    if (attn_split_heuristic_ex(1, 1, 28, 4, 128, 8192, 152, ATTN_VARIANT_TCGEN05) != 64) return 10;
    if (attn_decode(0, 0, 0, 0, 0, 1, 28, 5, 128, 0.1f, 0) != ATTN_ERR_INVALID_ARG) return 6;
    if (attn_selftest_bounded_wait(0, 0) != ATTN_ERR_INVALID_ARG) return 7;
    printf("ok\n");
    return 0;
}
''')
    libdir = os.path.dirname(pkg.library_path())
    exe = tmp_path / "use_abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lattn_decode", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0 and res.stdout.strip() == "ok", (res.returncode, res.stderr)


def test_decode_attention_checks_its_tensors_before_any_call():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 8, 128)
    k = torch.zeros(1, 64, 2, 128, dtype=torch.float16)
    pos = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(TypeError):
        pkg.decode_attention(q.double(), k, k, pos)                    # q must be f32
    with pytest.raises(TypeError):
        pkg.decode_attention(q, k.float(), k.float(), pos)             # cache must be 16-bit
    with pytest.raises(TypeError):
        pkg.decode_attention(q, k, k.bfloat16(), pos)                  # K and V of one type
    with pytest.raises(ValueError):
        pkg.decode_attention(q[:, :, :64], k, k, pos)                  # head_dim mismatch
    with pytest.raises(ValueError):
        pkg.decode_attention(q, k.transpose(1, 2), k.transpose(1, 2), pos)   # not contiguous
    with pytest.raises(ValueError):
        pkg.decode_attention(q, k, k, pos, kernel=9)                   # no such kernel


def test_tcgen05_choice_keeps_its_limits(lib):
    """Wherever variant 0 names a one-tile kernel (tcgen05, or the one-tile
    mma.sync kernel), the planned splits cover the capacity one tile each and
    fit one wave of its blocks; several query rows on the mma.sync form only at
    head_dim 128, on tcgen05 only when a KV head's pairs fit one 16-slot block.
    Seeded random shapes."""
    rng = np.random.default_rng(12)
    T5, VT = pkg.ATTN_VARIANT_TCGEN05, pkg.ATTN_VARIANT_TC_TILE
    tile = {128: 128, 256: 96}
    per_sm = {(128, False): 3, (256, False): 2, (128, True): 2, (256, True): 1}
    seen = set()
    for _ in range(4000):
        hd = int(rng.choice([64, 128, 256]))
        n_kv = int(rng.integers(1, 9))
        G = int(rng.integers(1, 9))
        n_q = int(rng.choice([1, 1, 2, 3, 4]))
        n_seq = int(rng.integers(1, 5))
        cap = int(rng.integers(1, 40000))
        sms = int(rng.choice([132, 148, 152]))
        flags = int(rng.choice([0, pkg.ATTN_KV_STABLE]))
        v = pkg.attn_resolve_variant(n_seq, n_q, G * n_kv, n_kv, hd, cap, sms, flags)
        P = pkg.attn_split_heuristic_ex(n_seq, n_q, G * n_kv, n_kv, hd, cap, sms, flags)
        assert v in (pkg.ATTN_VARIANT_TC, T5, VT) and P > 0
        if v not in (T5, VT):
            continue
        seen.add((hd, n_q > 1))
        assert hd in (128, 256)
        # the one-tile kernel may take its wide tiles (one block per SM): 256 rows at
        # head_dim 128, 128 at 256
        assert P * ((256 if hd == 128 else 128) if v == VT else tile[hd]) >= cap
        if v == VT:
            # 16 (row, head) slots per block; 3 blocks per SM at head_dim 128, 2 at 256
            assert n_q == 1 or hd == 128
            qg = 1 if n_q == 1 else -(-n_q * G // 16)
            assert P * n_kv * n_seq * qg <= sms * (3 if hd == 128 else 2)
        else:
            assert n_q == 1 or n_q * G <= 16
            assert P * n_kv * n_seq <= sms * per_sm[(hd, n_q > 1)]
    assert seen == {(128, False), (256, False), (128, True), (256, True)}
