"""Seeded synthetic workloads for decode attention.

This module only draws random inputs and describes workload shapes; it holds
none of the attention arithmetic. The same bytes it produces feed the CUDA
library (after a copy to the device) and the CPU oracle.

Recipe (every workload): q ~ N(0, 1) drawn in float32; K and V ~ N(0, 1)
drawn in float32, multiplied by ``k_scale`` (K only) and rounded to IEEE
binary16 with round-to-nearest-even (numpy's float32 -> float16 cast), or to
bfloat16 (round-to-nearest-even on the bit pattern) for a bfloat16 cache.
Each (workload, layer, sequence) pair draws from its own PCG64 stream seeded
with ``[seed, layer, sequence]``, so any slice can be regenerated alone.
Cache rows at or past a sequence's context length are never read by the
method; they are filled with ``fill`` (0 by default, NaN in tests that prove
those rows are ignored).

Shapes follow the workloads of the pages: the 7B decode of the minfer log
(28 query / 4 KV heads, head_dim 128, 2K context), the Qwen3-Next-like
long-context decode of Red Lite dev35 (16 / 2 heads, head_dim 256, ~8400
positions, 12 layers) and the hidden=32 / head_dim=8 fixture of dotLLM #199.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    n_seq: int
    n_head: int
    n_kv_head: int
    head_dim: int
    cap: int                      # cache rows allocated per sequence
    ctx: tuple                    # context length per sequence (positions = ctx - 1)
    layers: int = 1
    seed: int = 0
    k_scale: float = 1.0
    n_splits: int = 0             # 0 = let the library choose
    split_len: int = 0            # 0 = split by count
    scale: float = field(default=0.0)

    def __post_init__(self):
        if self.scale == 0.0:
            object.__setattr__(self, "scale", 1.0 / math.sqrt(self.head_dim))

    @property
    def group(self) -> int:
        return self.n_head // self.n_kv_head

    def kv_bytes(self) -> int:
        """K+V bytes the method reads for one layer: sum_s nkv_s * n_kv * hd * 2 B * 2."""
        rows = sum(min(max(c, 0), self.cap) for c in self.ctx)
        return rows * self.n_kv_head * self.head_dim * 2 * 2

    def with_ctx(self, ctx) -> "Workload":
        if isinstance(ctx, int):
            ctx = (ctx,) * self.n_seq
        return replace(self, ctx=tuple(int(c) for c in ctx))


def _ragged_ctx(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64([seed, 0xC7C]))
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


WORKLOADS = {
    # 1 sequence, 8/2 heads, hd 128, context 512, 4 splits
    "tiny": Workload("tiny", 1, 8, 2, 128, 512, (512,), seed=0, n_splits=4),
    # 7B-like decode: 28/4 heads (group 7), hd 128, context swept, 28 layers, cap 8192
    "7b": Workload("7b", 1, 28, 4, 128, 8192, (8192,), layers=28, seed=1),
    # long-context grouped: 16/2 heads (group 8), hd 256, context 8400, 12 layers
    "long": Workload("long", 1, 16, 2, 256, 8400, (8400,), layers=12, seed=2),
    # batched ragged: 32 sequences, context ~ U[1, 32768], 32/8 heads, hd 128
    "ragged": Workload("ragged", 32, 32, 8, 128, 32768, _ragged_ctx(3, 32, 1, 32768), seed=3),
    # stress: context 131072, 64/8 heads, hd 128, K x8
    "stress": Workload("stress", 1, 64, 8, 128, 131072, (131072,), seed=4, k_scale=8.0),
    # small-head fixture: 4/2 heads, hd 8, context 64
    "smallhead": Workload("smallhead", 1, 4, 2, 8, 64, (64,), seed=5),
}

CTX_SWEEP_7B = (128, 512, 2048, 8192)
BLOCK_SWEEP_LONG = (32, 64, 128, 256)


def _rng(seed: int, layer: int, seq: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, layer, seq, stream]))


def make_q(w: Workload, layer: int = 0) -> np.ndarray:
    """q: float32 [n_seq, n_head, head_dim]."""
    out = np.empty((w.n_seq, w.n_head, w.head_dim), dtype=np.float32)
    for s in range(w.n_seq):
        out[s] = _rng(w.seed, layer, s, 0).standard_normal(
            (w.n_head, w.head_dim), dtype=np.float32)
    return out


def make_q_multi(w: Workload, n_q: int, layer: int = 0) -> np.ndarray:
    """q for n_q causal query rows: float32 [n_seq, n_q, n_head, head_dim]."""
    out = np.empty((w.n_seq, n_q, w.n_head, w.head_dim), dtype=np.float32)
    for s in range(w.n_seq):
        out[s] = _rng(w.seed, layer, s, 3).standard_normal(
            (n_q, w.n_head, w.head_dim), dtype=np.float32)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def _cast(x: np.ndarray, kv_dtype: str) -> np.ndarray:
    return x.astype(np.float16) if kv_dtype == "f16" else to_bf16_bits(x)


def fill_kv_seq(w: Workload, layer: int, s: int, k_out: np.ndarray, v_out: np.ndarray,
                fill: float = 0.0, kv_dtype: str = "f16") -> None:
    """Fill one sequence's cache rows, k_out/v_out [cap, n_kv_head, head_dim]:
    float16, or bfloat16 bit patterns (uint16) for kv_dtype "bf16"."""
    n = min(max(w.ctx[s], 0), w.cap)
    shape = (n, w.n_kv_head, w.head_dim)
    k = _rng(w.seed, layer, s, 1).standard_normal(shape, dtype=np.float32)
    if w.k_scale != 1.0:
        k *= np.float32(w.k_scale)
    k_out[:n] = _cast(k, kv_dtype)
    del k
    v_out[:n] = _cast(_rng(w.seed, layer, s, 2).standard_normal(shape, dtype=np.float32), kv_dtype)
    if n < w.cap:
        f = _cast(np.full(1, fill, np.float32), kv_dtype)[0]
        k_out[n:] = f
        v_out[n:] = f


def make_kv(w: Workload, layer: int = 0, fill: float = 0.0, kv_dtype: str = "f16",
            threads: int = 1):
    """K, V [n_seq, cap, n_kv_head, head_dim]: float16, or bfloat16 bit
    patterns (uint16) for kv_dtype "bf16". With threads > 1 the sequences are
    drawn in parallel; every sequence has its own stream, so the bytes do not
    depend on the thread count."""
    shape = (w.n_seq, w.cap, w.n_kv_head, w.head_dim)
    dt = np.float16 if kv_dtype == "f16" else np.uint16
    k = np.empty(shape, dtype=dt)
    v = np.empty(shape, dtype=dt)
    if threads > 1 and w.n_seq > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(threads, w.n_seq)) as ex:
            list(ex.map(lambda s: fill_kv_seq(w, layer, s, k[s], v[s], fill, kv_dtype),
                        range(w.n_seq)))
    else:
        for s in range(w.n_seq):
            fill_kv_seq(w, layer, s, k[s], v[s], fill, kv_dtype)
    return k, v


def make_positions(w: Workload) -> np.ndarray:
    """positions[s] = ctx[s] - 1 (index of the current token), int32."""
    return np.asarray([c - 1 for c in w.ctx], dtype=np.int32)


def make_new_rows(w: Workload, layer: int = 0, kv_dtype: str = "f16"):
    """The new token's K and V rows for a fused append, [n_seq, n_kv_head,
    head_dim] each, in the cache's element type."""
    shape = (w.n_seq, w.n_kv_head, w.head_dim)
    kn = np.empty(shape, dtype=np.float16 if kv_dtype == "f16" else np.uint16)
    vn = np.empty_like(kn)
    for s in range(w.n_seq):
        kn[s] = _cast(_rng(w.seed, layer, s, 4).standard_normal(shape[1:], dtype=np.float32), kv_dtype)
        vn[s] = _cast(_rng(w.seed, layer, s, 5).standard_normal(shape[1:], dtype=np.float32), kv_dtype)
    return kn, vn


def make_layer(w: Workload, layer: int = 0, fill: float = 0.0, kv_dtype: str = "f16",
               threads: int = 1) -> dict:
    k, v = make_kv(w, layer, fill, kv_dtype, threads)
    return {"q": make_q(w, layer), "k": k, "v": v, "positions": make_positions(w)}
