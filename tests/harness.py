"""Shared helpers for the GPU tests: move seeded inputs to the device, call the
library through its C ABI, and compare element by element with the oracle.

Tolerance (f32 q, f32 accumulation over an f16 cache): per element
|gpu - oracle| <= 1e-4 + 1e-3 * |oracle|, the AbsTol(1e-4) + RelTol(1e-3) bar of
dotLLM issue #199 §0.
"""
import numpy as np

ABS_TOL = 1e-4
REL_TOL = 1e-3


def assert_close(got, ref, what="", abs_tol=ABS_TOL, rel_tol=REL_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = abs_tol + rel_tol * np.abs(ref)
    bad = ~(err <= bound)                      # NaN counts as a failure
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err, -1.0)), err.shape)
        raise AssertionError("%s: %d of %d elements outside %.0e + %.0e|ref|; worst at %s: got %r "
                             "want %r" % (what, int(bad.sum()), bad.size, abs_tol, rel_tol, idx,
                                          float(got[idx]), float(ref[idx])))
    return float(err.max()) if err.size else 0.0


def to_device(layer, device="cuda"):
    """numpy arrays -> device tensors; uint16 (bfloat16 bit patterns) travel as int16."""
    import torch
    out = {}
    for name, arr in layer.items():
        arr = np.ascontiguousarray(arr)
        if arr.dtype == np.uint16:
            arr = arr.view(np.int16)
        out[name] = torch.from_numpy(arr).to(device)
    return out


def run_decode(pkg, dev, n_head, n_kv_head, head_dim, cap, scale, n_splits=0, split_len=0,
               variant=0, workspace=None, stream=None):
    """Call attn_decode_ex on device tensors {q, k, v, positions}; returns out (torch)."""
    import torch
    out = torch.full_like(dev["q"], float("nan"))
    n_seq = dev["positions"].shape[0]
    pkg.attn_decode_ex(dev["q"], dev["k"], dev["v"], dev["positions"], out, n_seq, n_head,
                       n_kv_head, head_dim, scale, cap, n_splits=n_splits, split_len=split_len,
                       variant=variant, workspace=workspace, stream=stream)
    return out


def make_case(seed, n_seq, n_head, n_kv_head, head_dim, cap, ctx, k_scale=1.0, fill=0.0,
              kv_dtype="f16"):
    """Seeded inputs (q ~ N(0,1) f32; K, V ~ N(0,1) rounded to f16, or to bfloat16
    bit patterns for kv_dtype "bf16"), rows >= ctx set to `fill`."""
    from decode_attention_gqa_gb300.synthetic import to_bf16_bits
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((n_seq, n_head, head_dim), dtype=np.float32)
    k = rng.standard_normal((n_seq, cap, n_kv_head, head_dim), dtype=np.float32) * np.float32(k_scale)
    v = rng.standard_normal((n_seq, cap, n_kv_head, head_dim), dtype=np.float32)
    ctx = [int(c) for c in ctx]
    for s, c in enumerate(ctx):
        c = max(0, min(c, cap))
        k[s, c:] = fill
        v[s, c:] = fill
    if kv_dtype == "f16":
        k, v = k.astype(np.float16), v.astype(np.float16)
    else:
        k, v = to_bf16_bits(k), to_bf16_bits(v)
    positions = np.asarray(ctx, dtype=np.int32) - 1
    return {"q": q, "k": k, "v": v, "positions": positions}
