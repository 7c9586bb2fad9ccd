"""GB300 (sm_103a) split-KV grouped-query decode attention.

Thin ctypes binding over ``libattn_decode.so`` (declared in
``include/attn_decode.h``). Every function here has the name and argument order
of the C entry point it calls and does argument marshalling only: pointers may
be given as integers or as tensors (their ``data_ptr()`` is passed), streams as
integers, ``torch.cuda.Stream`` objects or ``None`` (the current torch stream).
All arithmetic runs in the library's CUDA kernels; if the library has not been
built, every call raises ``RuntimeError`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "AttnError", "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_WORKSPACE",
    "ATTN_ERR_CUDA", "ATTN_DEVERR_POSITION_CLAMPED", "ATTN_DEVERR_PIPELINE_TIMEOUT",
    "ATTN_VARIANT_AUTO", "ATTN_VARIANT_SIMT", "ATTN_VARIANT_TC", "ATTN_VARIANT_TCGEN05",
    "ATTN_VARIANT_TCGEN05_CLUSTER", "ATTN_VARIANT_TC_TILE", "ATTN_KV_BF16",
    "ATTN_KV_STABLE",
    "library_path",
    "load",
    "attn_decode", "attn_decode_ex", "attn_decode_append", "attn_decode_multi", "decode_attention",
    "attn_decode_partial",
    "attn_decode_combine",
    "attn_decode_static",
    "attn_split_heuristic", "attn_split_heuristic_ex", "attn_resolve_variant", "attn_plan_call",
    "attn_workspace_size",
    "attn_read_device_error", "attn_selftest_bounded_wait", "attn_status_string",
    "attn_last_cuda_error", "attn_version",
]

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA = range(5)
ATTN_DEVERR_POSITION_CLAMPED = 0x1
ATTN_DEVERR_PIPELINE_TIMEOUT = 0x2
ATTN_VARIANT_AUTO, ATTN_VARIANT_SIMT, ATTN_VARIANT_TC, ATTN_VARIANT_TCGEN05 = 0, 1, 2, 3
ATTN_VARIANT_TCGEN05_CLUSTER = 4
ATTN_VARIANT_TC_TILE = 5
ATTN_KV_BF16 = 0x10
ATTN_KV_STABLE = 0x20

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = attn_status_string(status)
        extra = ""
        if status == ATTN_ERR_CUDA:
            extra = " (cudaError %d)" % attn_last_cuda_error()
        super().__init__("%s returned %s%s" % (where, name, extra))


def library_path() -> str:
    return os.path.join(_PKG, "libattn_decode.so")


def load():
    """Load the library (once). Raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libattn_decode.so is not built (%s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.attn_decode.restype = i32
        lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp]
        lib.attn_decode_ex.restype = i32
        lib.attn_decode_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i64, i32, i32,
                                       i32, vp, sz, vp]
        lib.attn_decode_append.restype = i32
        lib.attn_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i64,
                                           i32, i32, i32, vp, sz, vp]
        lib.attn_decode_multi.restype = i32
        lib.attn_decode_multi.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i64, i32,
                                          i32, i32, vp, sz, vp]
        lib.attn_decode_partial.restype = i32
        lib.attn_decode_partial.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, i64, i32, i32,
                                            i32, vp, sz, vp]
        lib.attn_decode_combine.restype = i32
        lib.attn_decode_combine.argtypes = [vp, sz, vp, i32, i32, i32, i32, vp]
        lib.attn_decode_static.restype = i32
        lib.attn_decode_static.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i64, i32,
                                           i32, i32, vp]
        lib.attn_split_heuristic.restype = i32
        lib.attn_split_heuristic.argtypes = [i32, i32, i32, i32, i64, i32]
        lib.attn_split_heuristic_ex.restype = i32
        lib.attn_split_heuristic_ex.argtypes = [i32, i32, i32, i32, i32, i64, i32, i32]
        lib.attn_resolve_variant.restype = i32
        lib.attn_resolve_variant.argtypes = [i32, i32, i32, i32, i32, i64, i32, i32]
        lib.attn_plan_call.restype = i32
        lib.attn_plan_call.argtypes = [i32, i32, i32, i32, i32, i64, i32, i32, i32,
                                       ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(sz)]
        lib.attn_workspace_size.restype = sz
        lib.attn_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.attn_read_device_error.restype = i32
        lib.attn_read_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        lib.attn_selftest_bounded_wait.restype = i32
        lib.attn_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i32]
        lib.attn_last_cuda_error.restype = i32
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_version.restype = i32
        lib.attn_version.argtypes = []
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError("expected an int address or a tensor, got %r" % type(x))


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError("expected a stream handle, torch.cuda.Stream or None")


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_decode(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim, scale,
                stream=None):
    """o = softmax(q·Kᵀ·scale)·V for one sequence (see include/attn_decode.h)."""
    _check(load().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions), _ptr(out),
                              n_seq, n_head, n_kv_head, head_dim, scale, _stream(stream)),
           "attn_decode")


def attn_decode_ex(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim, scale,
                   cap, n_splits=0, split_len=0, variant=ATTN_VARIANT_AUTO, workspace=None,
                   workspace_bytes=0, stream=None):
    """Several sequences, explicit capacity, split and workspace control."""
    if workspace is not None and not workspace_bytes and hasattr(workspace, "nbytes"):
        workspace_bytes = workspace.nbytes
    _check(load().attn_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions), _ptr(out),
                                 n_seq, n_head, n_kv_head, head_dim, scale, cap, n_splits,
                                 split_len, variant, _ptr(workspace), workspace_bytes,
                                 _stream(stream)),
           "attn_decode_ex")


def decode_attention(q, k_cache, v_cache, positions, scale=None, out=None, n_splits=0,
                     kv_stable=False, stream=None, kernel=ATTN_VARIANT_AUTO):
    """Convenience form of attn_decode_ex for torch tensors: the sizes come
    from the shapes -- q f32 [n_seq, n_head, head_dim] (or [n_seq, n_q,
    n_head, head_dim] for several causal query rows, attn_decode_multi),
    k_cache / v_cache float16 or bfloat16 [n_seq, cap, n_kv_head, head_dim],
    positions int32 [n_seq] -- scale defaults to 1/sqrt(head_dim), the cache
    dtype picks ATTN_KV_BF16, and `out` is allocated when not given. `kernel`
    is one of the ATTN_VARIANT_* values (variant 0, the library's choice, by
    default). The library-owned workspace is used. Returns out."""
    import math
    import torch
    if q.dtype != torch.float32 or positions.dtype != torch.int32:
        raise TypeError("q must be float32 and positions int32")
    if k_cache.dtype != v_cache.dtype or k_cache.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("k_cache and v_cache must both be float16 or both bfloat16")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache / v_cache must be [n_seq, cap, n_kv_head, head_dim]")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("positions", positions)):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    n_seq, cap, n_kv_head, head_dim = k_cache.shape
    if q.dim() == 3:
        n_q, (qs, n_head, qd) = 1, q.shape
    elif q.dim() == 4:
        qs, n_q, n_head, qd = q.shape
    else:
        raise ValueError("q must be [n_seq, n_head, head_dim] or [n_seq, n_q, n_head, head_dim]")
    if qs != n_seq or qd != head_dim or positions.numel() != n_seq:
        raise ValueError("q, the caches and positions disagree on n_seq or head_dim")
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    if kernel not in (ATTN_VARIANT_AUTO, ATTN_VARIANT_SIMT, ATTN_VARIANT_TC, ATTN_VARIANT_TCGEN05,
                      ATTN_VARIANT_TCGEN05_CLUSTER, ATTN_VARIANT_TC_TILE):
        raise ValueError("kernel must be one of the ATTN_VARIANT_* values")
    variant = kernel | (ATTN_KV_BF16 if k_cache.dtype == torch.bfloat16 else 0) | \
        (ATTN_KV_STABLE if kv_stable else 0)
    if n_q > 1:
        attn_decode_multi(q, k_cache, v_cache, positions, out, n_seq, n_q, n_head, n_kv_head,
                          head_dim, scale, cap, n_splits=n_splits, variant=variant, stream=stream)
    else:
        attn_decode_ex(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, cap, n_splits=n_splits, variant=variant, stream=stream)
    return out


def attn_decode_append(q, k_new, v_new, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head,
                       head_dim, scale, cap, n_splits=0, split_len=0, variant=ATTN_VARIANT_AUTO,
                       workspace=None, workspace_bytes=0, stream=None):
    """Write the new token's K/V row at positions[s] and attend, fused."""
    if workspace is not None and not workspace_bytes and hasattr(workspace, "nbytes"):
        workspace_bytes = workspace.nbytes
    _check(load().attn_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(positions), _ptr(out), n_seq, n_head,
                                     n_kv_head, head_dim, scale, cap, n_splits, split_len, variant,
                                     _ptr(workspace), workspace_bytes, _stream(stream)),
           "attn_decode_append")


def attn_decode_multi(q, k_cache, v_cache, positions, out, n_seq, n_q, n_head, n_kv_head, head_dim,
                      scale, cap, n_splits=0, split_len=0, variant=ATTN_VARIANT_AUTO,
                      workspace=None, workspace_bytes=0, stream=None):
    """n_q causal query rows per sequence (see include/attn_decode.h)."""
    if workspace is not None and not workspace_bytes and hasattr(workspace, "nbytes"):
        workspace_bytes = workspace.nbytes
    _check(load().attn_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions),
                                    _ptr(out), n_seq, n_q, n_head, n_kv_head, head_dim, scale, cap,
                                    n_splits, split_len, variant, _ptr(workspace), workspace_bytes,
                                    _stream(stream)),
           "attn_decode_multi")


def attn_decode_partial(q, k_cache, v_cache, positions, n_seq, n_head, n_kv_head, head_dim,
                        scale, cap, n_splits, split_len=0, variant=ATTN_VARIANT_AUTO,
                        workspace=None, workspace_bytes=0, stream=None):
    """Stage one (partials into `workspace`); see include/attn_decode.h."""
    if workspace is not None and not workspace_bytes and hasattr(workspace, "nbytes"):
        workspace_bytes = workspace.nbytes
    _check(load().attn_decode_partial(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions),
                                      n_seq, n_head, n_kv_head, head_dim, scale, cap, n_splits,
                                      split_len, variant, _ptr(workspace), workspace_bytes,
                                      _stream(stream)),
           "attn_decode_partial")


def attn_decode_combine(workspace, workspace_bytes, out, n_seq, n_head, head_dim, n_splits,
                        stream=None):
    """Stage two (combine the partials in `workspace` into `out`)."""
    if not workspace_bytes and hasattr(workspace, "nbytes"):
        workspace_bytes = workspace.nbytes
    _check(load().attn_decode_combine(_ptr(workspace), workspace_bytes, _ptr(out), n_seq, n_head,
                                      head_dim, n_splits, _stream(stream)),
           "attn_decode_combine")


def attn_decode_static(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, cap, n_splits=0, split_len=0, variant=ATTN_VARIANT_AUTO, stream=None):
    """attn_decode_ex with the library's fixed scratch array instead of a
    workspace: allocates nothing (see include/attn_decode.h)."""
    _check(load().attn_decode_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions),
                                     _ptr(out), n_seq, n_head, n_kv_head, head_dim, scale, cap,
                                     n_splits, split_len, variant, _stream(stream)),
           "attn_decode_static")


def attn_split_heuristic(n_seq, n_head, n_kv_head, head_dim, cap, sm_count) -> int:
    return load().attn_split_heuristic(n_seq, n_head, n_kv_head, head_dim, cap, sm_count)


def attn_split_heuristic_ex(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count, variant) -> int:
    return load().attn_split_heuristic_ex(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count,
                                          variant)


def attn_resolve_variant(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count, variant) -> int:
    """The partial kernel (ATTN_VARIANT_SIMT / _TC / _TCGEN05) such a call runs with
    the heuristic's split count; 0 for an unsupported shape."""
    return load().attn_resolve_variant(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count,
                                       variant)


def attn_plan_call(n_seq, n_q, n_head, n_kv_head, head_dim, cap, n_splits=0, split_len=0,
                   variant=0):
    """(kernel variant, split count, workspace bytes) of the call with these
    arguments; raises AttnError with the status the call would return."""
    v = ctypes.c_int(0)
    p = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    _check(load().attn_plan_call(n_seq, n_q, n_head, n_kv_head, head_dim, cap, n_splits, split_len,
                                 variant, ctypes.byref(v), ctypes.byref(p), ctypes.byref(ws)),
           "attn_plan_call")
    return v.value, p.value, ws.value


def attn_workspace_size(n_seq, n_head, head_dim, n_splits) -> int:
    return load().attn_workspace_size(n_seq, n_head, head_dim, n_splits)


def attn_selftest_bounded_wait(limit_ns, stream=None) -> None:
    """Launch the bounded-wait self-test (see include/attn_decode.h)."""
    _check(load().attn_selftest_bounded_wait(limit_ns, _stream(stream)),
           "attn_selftest_bounded_wait")


def attn_read_device_error(stream=None) -> int:
    flags = ctypes.c_uint(0)
    _check(load().attn_read_device_error(_stream(stream), ctypes.byref(flags)),
           "attn_read_device_error")
    return flags.value


def attn_status_string(status) -> str:
    return load().attn_status_string(status).decode()


def attn_last_cuda_error() -> int:
    return load().attn_last_cuda_error()


def attn_version() -> int:
    return load().attn_version()
