"""Double-precision CPU oracle for split-KV grouped-query decode attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package. The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, its own
binary16 decoder). This module compiles it with gcc on first use and exposes
thin ctypes wrappers that take numpy arrays.

What it computes: o = softmax(q·Kᵀ·scale)·V per (sequence, query head), with
query head h reading KV head h // (n_head // n_kv_head) and the row count
nkv = clamp(positions[s] + 1, 0, cap) -- "10 · R4 -- decode split-attention
dim-parallel rewrite", §2.1 and §2.2 (minfer CUDA optimisation log).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags: tuple = ()) -> str:
    """Compile the oracle into a shared library with gcc (-O2, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    p = ctypes.c_void_p
    lib.oracle_f16_to_double.restype = dbl
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double_array.restype = None
    lib.oracle_f16_to_double_array.argtypes = [p, p, i64]
    lib.oracle_bf16_to_double_array.restype = None
    lib.oracle_bf16_to_double_array.argtypes = [p, p, i64]
    common = [p, p, p, p, p, i32, i32, i32, i32, i64, dbl]
    lib.oracle_attn_decode.restype = i32
    lib.oracle_attn_decode.argtypes = common + [i32]
    lib.oracle_attn_decode_one.restype = i32
    lib.oracle_attn_decode_one.argtypes = common + [i32, i32]
    lib.oracle_attn_decode_kv.restype = i32
    lib.oracle_attn_decode_kv.argtypes = common + [i32, i32]
    lib.oracle_attn_decode_one_kv.restype = i32
    lib.oracle_attn_decode_one_kv.argtypes = common + [i32, i32, i32]
    lib.oracle_attn_decode_multi.restype = i32
    lib.oracle_attn_decode_multi.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i64, dbl, i32,
                                             i32]
    lib.oracle_attn_decode_split.restype = i32
    lib.oracle_attn_decode_split.argtypes = common + [i32, i64]
    return lib


def load_library(path: str | None = None):
    """Load (building first if missing or older than the source) the oracle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _prep(q, k, v, positions):
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k).view(np.uint16)
    v = np.ascontiguousarray(v).view(np.uint16)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    return q, k, v, positions


KV_DTYPES = {"f16": 0, "bf16": 1}


def bf16_to_double(bits, lib=None) -> np.ndarray:
    """Decode an array of bfloat16 bit patterns (uint16) to float64."""
    lib = lib or load_library()
    b = np.ascontiguousarray(bits).view(np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_bf16_to_double_array(_ptr(b), _ptr(out), b.size)
    return out


def f16_to_double(bits, lib=None) -> np.ndarray:
    """Decode an array of binary16 bit patterns (uint16 or float16) to float64."""
    lib = lib or load_library()
    b = np.ascontiguousarray(bits).view(np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_f16_to_double_array(_ptr(b), _ptr(out), b.size)
    return out


def attn_decode(q, k, v, positions, n_head, n_kv_head, head_dim, cap, scale,
                n_threads=1, lib=None, kv_dtype="f16") -> np.ndarray:
    """Single-pass oracle over every (sequence, head).

    q: f32 [n_seq, n_head, head_dim]; k, v: f16, or 16-bit patterns of
    `kv_dtype` ("f16" or "bf16"), [n_seq, cap, n_kv_head, head_dim];
    positions: int32 [n_seq]. Returns float64 [n_seq, n_head, head_dim].
    """
    lib = lib or load_library()
    q, k, v, positions = _prep(q, k, v, positions)
    n_seq = positions.shape[0]
    out = np.zeros((n_seq, n_head, head_dim), dtype=np.float64)
    if kv_dtype == "f16":
        rc = lib.oracle_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(out),
                                    n_seq, n_head, n_kv_head, head_dim, cap, float(scale),
                                    int(n_threads))
    else:
        rc = lib.oracle_attn_decode_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(out),
                                       n_seq, n_head, n_kv_head, head_dim, cap, float(scale),
                                       int(n_threads), KV_DTYPES[kv_dtype])
    if rc != 0:
        raise ValueError("oracle_attn_decode failed with status %d" % rc)
    return out


def attn_decode_one(q, k, v, positions, n_head, n_kv_head, head_dim, cap, scale, s, h,
                    lib=None, kv_dtype="f16") -> np.ndarray:
    """One output row o[s, h, :] (float64), for sampled checks on big workloads."""
    lib = lib or load_library()
    q, k, v, positions = _prep(q, k, v, positions)
    out = np.zeros(head_dim, dtype=np.float64)
    rc = lib.oracle_attn_decode_one_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(out),
                                       positions.shape[0], n_head, n_kv_head, head_dim, cap,
                                       float(scale), int(s), int(h), KV_DTYPES[kv_dtype])
    if rc != 0:
        raise ValueError("oracle_attn_decode_one failed with status %d" % rc)
    return out


def attn_decode_split(q, k, v, positions, n_head, n_kv_head, head_dim, cap, scale,
                      n_splits, split_len=0, lib=None) -> np.ndarray:
    """Two-stage (partials + combine) restatement, float64 result."""
    lib = lib or load_library()
    q, k, v, positions = _prep(q, k, v, positions)
    n_seq = positions.shape[0]
    out = np.zeros((n_seq, n_head, head_dim), dtype=np.float64)
    rc = lib.oracle_attn_decode_split(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(out),
                                      n_seq, n_head, n_kv_head, head_dim, cap, float(scale),
                                      int(n_splits), int(split_len))
    if rc != 0:
        raise ValueError("oracle_attn_decode_split failed with status %d" % rc)
    return out


def attn_decode_multi(q, k, v, positions, n_q, n_head, n_kv_head, head_dim, cap, scale,
                      n_threads=1, lib=None, kv_dtype="f16") -> np.ndarray:
    """Causal multi-query oracle: q f32 [n_seq, n_q, n_head, head_dim]; query row t
    attends the first clamp(positions[s]+1, 0, cap) - n_q + t + 1 rows.
    Returns float64 [n_seq, n_q, n_head, head_dim]."""
    lib = lib or load_library()
    q, k, v, positions = _prep(q, k, v, positions)
    n_seq = positions.shape[0]
    out = np.zeros((n_seq, n_q, n_head, head_dim), dtype=np.float64)
    rc = lib.oracle_attn_decode_multi(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(out),
                                      n_seq, n_q, n_head, n_kv_head, head_dim, cap, float(scale),
                                      int(n_threads), KV_DTYPES[kv_dtype])
    if rc != 0:
        raise ValueError("oracle_attn_decode_multi failed with status %d" % rc)
    return out
