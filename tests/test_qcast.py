"""Host-side q-cast isolation check (dotLLM issue #199 §0, "Precondition
check"): before q goes to 16-bit tensor-core operands, measure on the CPU,
with the oracle alone, what rounding q does to the attention output.

- A single cast of q to binary16 (the design that issue's §2 ports) moves the
  output past the f32-q bar (1e-4 abs + 1e-3 rel) once scores spread widely
  (K scaled x8, as in the stress workload); that is why the issue allows a
  looser 5e-3 bar for a cast q.
- The pair the tensor-core kernel carries instead, hi = T(q) and
  lo = T(q - hi) for T the cache's element type, stays far inside the f32 bar
  for binary16 and inside it for bfloat16.

Everything here is numpy plus the oracle; no GPU code is involved."""
import numpy as np

import oracle
from harness import ABS_TOL, REL_TOL, make_case


def _excess(got, ref):
    """max over elements of |got - ref| / (ABS_TOL + REL_TOL |ref|): <= 1 passes the bar."""
    return float(np.max(np.abs(got - ref) / (ABS_TOL + REL_TOL * np.abs(ref))))


def _to_bf16(x):
    from decode_attention_gqa_gb300.synthetic import to_bf16_bits
    return (to_bf16_bits(x).astype(np.uint32) << 16).view(np.float32)


def _cases():
    n_head, n_kv, hd, cap = 28, 4, 128, 1024
    yield "N(0,1) K", make_case(1300, 1, n_head, n_kv, hd, cap, (1000,)), n_head, n_kv, hd, cap
    yield "K x8", make_case(1301, 1, n_head, n_kv, hd, cap, (1000,), k_scale=8.0), n_head, n_kv, hd, cap


def test_single_f16_cast_of_q_breaks_the_f32_bar_under_spread():
    worst = {}
    for name, c, n_head, n_kv, hd, cap in _cases():
        scale = 1 / np.sqrt(hd)
        ref = oracle.attn_decode(c["q"], c["k"], c["v"], c["positions"], n_head, n_kv, hd, cap,
                                 scale, n_threads=8)
        q16 = c["q"].astype(np.float16).astype(np.float32)
        got = oracle.attn_decode(q16, c["k"], c["v"], c["positions"], n_head, n_kv, hd, cap, scale,
                                 n_threads=8)
        worst[name] = _excess(got, ref)
    assert worst["K x8"] > 1.0, worst          # outside 1e-4 + 1e-3 |ref| somewhere
    assert worst["N(0,1) K"] < worst["K x8"], worst


def test_hi_lo_pairs_of_q_stay_inside_the_f32_bar():
    for name, c, n_head, n_kv, hd, cap in _cases():
        scale = 1 / np.sqrt(hd)
        ref = oracle.attn_decode(c["q"], c["k"], c["v"], c["positions"], n_head, n_kv, hd, cap,
                                 scale, n_threads=8)
        q = c["q"]
        # binary16: hi + lo carries about 22 significant bits of q
        hi = q.astype(np.float16).astype(np.float32)
        lo = (q - hi).astype(np.float16).astype(np.float32)
        got = oracle.attn_decode(hi + lo, c["k"], c["v"], c["positions"], n_head, n_kv, hd, cap,
                                 scale, n_threads=8)
        assert _excess(got, ref) < 0.05, (name, "f16 pair")
        # bfloat16: about 16 bits
        hib = _to_bf16(q)
        lob = _to_bf16(q - hib)
        got = oracle.attn_decode(hib + lob, c["k"], c["v"], c["positions"], n_head, n_kv, hd, cap,
                                 scale, n_threads=8)
        assert _excess(got, ref) < 1.0, (name, "bf16 pair")
