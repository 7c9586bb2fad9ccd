"""Pins for the CPU oracle (no GPU).

The oracle is trusted only because these tests tie it to things other than
itself: an exact binary16 decode from an independent library, a 50-digit
decimal brute force, closed forms (one row, constant K, constant V, scale 0),
invariants (row permutation, score shift, linearity in V, GQA head mapping,
unread rows) and the two-stage split restatement of "10 · R4 -- decode
split-attention dim-parallel rewrite" §2.1-§2.2. ``test_oracle_mutants.py``
plants mistakes in a copy of the oracle and checks these pins catch them.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from decode_attention_gqa_gb300 import synthetic as syn


def _case(rng, n_seq, n_head, n_kv, hd, cap, ctx, k_scale=1.0):
    q = rng.standard_normal((n_seq, n_head, hd), dtype=np.float32)
    k = (rng.standard_normal((n_seq, cap, n_kv, hd), dtype=np.float32) * k_scale).astype(np.float16)
    v = rng.standard_normal((n_seq, cap, n_kv, hd), dtype=np.float32).astype(np.float16)
    pos = np.asarray(ctx, dtype=np.int32) - 1
    return q, k, v, pos


def _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib=None):
    return oracle.attn_decode(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib=lib)


# ---------------------------------------------------------------- f16 decoding

def check_f16_decoder(lib=None):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_double(bits, lib=lib)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_decoder_all_patterns():
    check_f16_decoder()


def check_bf16_decoder(lib=None):
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_double(bits, lib=lib)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns():
    check_bf16_decoder()


def to_bf16_bits(x):
    """float32 array -> bfloat16 bit patterns (round to nearest even, via torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(b):
    import torch
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


# ------------------------------------------------------- 50-digit brute force

def decimal_attention(q, k, v, pos, n_head, n_kv, hd, cap, scale):
    """Full score matrix and softmax in 50-digit decimal arithmetic."""
    getcontext().prec = 50
    n_seq = q.shape[0]
    G = n_head // n_kv
    out = np.zeros((n_seq, n_head, hd))
    sc = Decimal(float(scale))
    for s in range(n_seq):
        n = max(0, min(int(pos[s]) + 1, cap))
        for h in range(n_head):
            if n == 0:
                continue
            hk = h // G
            qd = [Decimal(float(x)) for x in q[s, h]]
            scores = []
            for j in range(n):
                kd = [Decimal(float(x)) for x in k[s, j, hk].astype(np.float64)]
                scores.append(sc * sum(a * b for a, b in zip(qd, kd)))
            m = max(scores)
            w = [(x - m).exp() for x in scores]
            Z = sum(w)
            for d in range(hd):
                acc = sum(wj * Decimal(float(v[s, j, hk, d])) for j, wj in enumerate(w))
                out[s, h, d] = float(acc / Z)
    return out


def check_bruteforce(lib=None):
    rng = np.random.Generator(np.random.PCG64(11))
    for (n_seq, n_head, n_kv, hd, cap, ctx) in [
        (1, 4, 2, 8, 16, (16,)),
        (2, 4, 1, 8, 12, (5, 12)),
        (1, 3, 3, 8, 9, (9,)),
        (2, 6, 2, 8, 7, (0, 7)),
    ]:
        q, k, v, pos = _case(rng, n_seq, n_head, n_kv, hd, cap, ctx)
        scale = 1.0 / math.sqrt(hd)
        got = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
        ref = decimal_attention(q, k, v, pos, n_head, n_kv, hd, cap, scale)
        assert np.max(np.abs(got - ref)) <= 1e-13


def test_bruteforce_decimal():
    check_bruteforce()


def check_bruteforce_bf16(lib=None):
    """The bfloat16 entry points against the same 50-digit brute force."""
    pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(21))
    for (n_seq, n_head, n_kv, hd, cap, ctx) in [(1, 4, 2, 8, 12, (12,)), (2, 6, 3, 8, 9, (4, 9))]:
        q = rng.standard_normal((n_seq, n_head, hd), dtype=np.float32)
        kb = to_bf16_bits(rng.standard_normal((n_seq, cap, n_kv, hd), dtype=np.float32) * 3)
        vb = to_bf16_bits(rng.standard_normal((n_seq, cap, n_kv, hd), dtype=np.float32))
        pos = np.asarray(ctx, np.int32) - 1
        scale = 1.0 / math.sqrt(hd)
        got = oracle.attn_decode(q, kb, vb, pos, n_head, n_kv, hd, cap, scale, lib=lib,
                                 kv_dtype="bf16")
        ref = decimal_attention(q, bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), pos, n_head, n_kv,
                                hd, cap, scale)
        assert np.max(np.abs(got - ref)) <= 1e-13
        one = oracle.attn_decode_one(q, kb, vb, pos, n_head, n_kv, hd, cap, scale, n_seq - 1,
                                     n_head - 1, lib=lib, kv_dtype="bf16")
        assert np.array_equal(one, got[n_seq - 1, n_head - 1])


def test_bruteforce_decimal_bf16():
    check_bruteforce_bf16()


# ------------------------------------------------------------- closed forms

def check_closed_forms(lib=None):
    rng = np.random.Generator(np.random.PCG64(12))
    n_head, n_kv, hd, cap = 8, 2, 128, 40
    scale = 1.0 / math.sqrt(hd)
    # one row: o is exactly that V row
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (1,))
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    for h in range(n_head):
        assert np.array_equal(o[0, h], v[0, 0, h // 4].astype(np.float64))
    # constant K rows: uniform weights, o is the mean of the V rows
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (37,))
    k[:] = k[:, :1]
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    mean = v[0, :37].astype(np.float64).mean(axis=0)
    for h in range(n_head):
        assert np.max(np.abs(o[0, h] - mean[h // 4])) <= 1e-14
    # scale 0: uniform weights as well
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (29,))
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, 0.0, lib)
    mean = v[0, :29].astype(np.float64).mean(axis=0)
    for h in range(n_head):
        assert np.max(np.abs(o[0, h] - mean[h // 4])) <= 1e-14
    # constant V rows: o equals that row whatever the weights
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (33,))
    v[:] = v[:, :1]
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    for h in range(n_head):
        assert np.max(np.abs(o[0, h] - v[0, 0, h // 4].astype(np.float64))) <= 1e-14
    # two rows with a known score gap: o = (v0 + e^g v1) / (1 + e^g)
    q = np.zeros((1, 1, 8), np.float32)
    q[0, 0, 0] = 1.0
    k = np.zeros((1, 2, 1, 8), np.float16)
    k[0, 1, 0, 0] = 0.75                       # score gap 0.75 * scale, scale = 2
    v = np.zeros((1, 2, 1, 8), np.float16)
    v[0, 0, 0, :] = 1.0
    v[0, 1, 0, :] = -3.0
    o = _run(q, k, v, np.array([1], np.int32), 1, 1, 8, 2, 2.0, lib)
    e = math.exp(1.5)
    assert np.max(np.abs(o[0, 0] - (1.0 - 3.0 * e) / (1.0 + e))) <= 1e-15


def test_closed_forms():
    check_closed_forms()


# --------------------------------------------------------------- invariants

def check_invariants(lib=None):
    rng = np.random.Generator(np.random.PCG64(13))
    n_head, n_kv, hd, cap = 8, 2, 64, 50
    scale = 1.0 / math.sqrt(hd)
    q, k, v, pos = _case(rng, 2, n_head, n_kv, hd, cap, (50, 23))
    base = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    assert np.all(np.isfinite(base))
    # permuting the live rows of one sequence leaves its output unchanged
    perm = rng.permutation(23)
    k2, v2 = k.copy(), v.copy()
    k2[1, :23] = k[1, perm]
    v2[1, :23] = v[1, perm]
    o = _run(q, k2, v2, pos, n_head, n_kv, hd, cap, scale, lib)
    assert np.max(np.abs(o - base)) <= 1e-14
    # linearity in V: doubling V (exact in f16 here) doubles o exactly
    o = _run(q, k, (v.astype(np.float32) * 2).astype(np.float16), pos, n_head, n_kv, hd, cap,
             scale, lib)
    assert np.array_equal(o, 2 * base)
    # shift invariance: a dimension where q is 1 and every K row holds the same
    # value adds one constant to all scores of a head
    q3 = q.copy()
    k3 = k.copy()
    q3[:, :, 0] = 1.0
    k3[:, :, :, 0] = np.float16(3.0)
    ref = _run(q3, k3, v, pos, n_head, n_kv, hd, cap, scale, lib)
    k3[:, :, :, 0] = np.float16(-5.0)
    o = _run(q3, k3, v, pos, n_head, n_kv, hd, cap, scale, lib)
    assert np.max(np.abs(o - ref)) <= 1e-13
    # rows at or past nkv are never read: NaN there changes nothing
    k4, v4 = k.copy(), v.copy()
    k4[1, 23:] = np.nan
    v4[1, 23:] = np.nan
    o = _run(q, k4, v4, pos, n_head, n_kv, hd, cap, scale, lib)
    assert np.array_equal(o, base)


def test_invariants():
    check_invariants()


def check_gqa_mapping(lib=None):
    rng = np.random.Generator(np.random.PCG64(14))
    n_head, n_kv, hd, cap = 8, 2, 16, 20
    G = n_head // n_kv
    scale = 0.3
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (17,))
    gqa = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    # MHA with each KV head replicated G times gives the same result
    k_mha = np.repeat(k, G, axis=2)
    v_mha = np.repeat(v, G, axis=2)
    mha = _run(q, k_mha, v_mha, pos, n_head, n_head, hd, cap, scale, lib)
    assert np.array_equal(gqa, mha)
    # MQA: each head alone against the single KV head
    mqa = _run(q, k[:, :, :1], v[:, :, :1], pos, n_head, 1, hd, cap, scale, lib)
    for h in range(n_head):
        one = _run(q[:, h:h + 1], k[:, :, :1], v[:, :, :1], pos, 1, 1, hd, cap, scale, lib)
        assert np.array_equal(mqa[:, h], one[:, 0])
    # swapping the two KV heads swaps which query-head group sees which cache
    sw = _run(q[:, np.r_[G:2 * G, 0:G]], k[:, :, ::-1], v[:, :, ::-1], pos, n_head, n_kv, hd,
              cap, scale, lib)
    assert np.array_equal(sw, gqa[:, np.r_[G:2 * G, 0:G]])


def test_gqa_mapping():
    check_gqa_mapping()


def check_positions(lib=None):
    rng = np.random.Generator(np.random.PCG64(15))
    n_head, n_kv, hd, cap = 4, 2, 8, 10
    q, k, v, _ = _case(rng, 4, n_head, n_kv, hd, cap, (1, 1, 1, 1))
    pos = np.array([-1, cap - 1, cap + 100, -(2 ** 31)], np.int32)
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, 0.5, lib)
    assert np.array_equal(o[0], np.zeros_like(o[0]))        # nkv = 0 -> 0
    assert np.array_equal(o[3], np.zeros_like(o[3]))
    # past the cache: clamped to cap rows, same as positions = cap - 1
    q2 = q.copy()
    q2[2] = q[1]
    k2, v2 = k.copy(), v.copy()
    k2[2], v2[2] = k[1], v[1]
    o2 = _run(q2, k2, v2, pos, n_head, n_kv, hd, cap, 0.5, lib)
    assert np.array_equal(o2[2], o2[1])


def test_positions_edges():
    check_positions()


# ------------------------------------------- two-stage split restatement

def check_split_equivalence(lib=None):
    rng = np.random.Generator(np.random.PCG64(16))
    n_head, n_kv, hd, cap = 8, 2, 32, 70
    ctx = (70, 33, 1, 0)
    q, k, v, pos = _case(rng, 4, n_head, n_kv, hd, cap, ctx, k_scale=3.0)
    scale = 1.0 / math.sqrt(hd)
    single = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    for P in (1, 2, 3, 7, 32, 70, 75):
        two = oracle.attn_decode_split(q, k, v, pos, n_head, n_kv, hd, cap, scale, P, lib=lib)
        assert np.max(np.abs(two - single)) <= 1e-12, P
    for blk in (1, 8, 16, 64):
        P = -(-cap // blk)
        two = oracle.attn_decode_split(q, k, v, pos, n_head, n_kv, hd, cap, scale, P, blk,
                                       lib=lib)
        assert np.max(np.abs(two - single)) <= 1e-12, blk


def test_split_equivalence():
    check_split_equivalence()


# ------------------------------------------------------------- stability

def check_stability(lib=None):
    """Large score spread (K x8, as in the stress workload) stays finite, and a
    planted row aligned with q takes all the weight."""
    rng = np.random.Generator(np.random.PCG64(17))
    n_head, n_kv, hd, cap = 8, 1, 128, 300
    q, k, v, pos = _case(rng, 1, n_head, n_kv, hd, cap, (300,), k_scale=8.0)
    scale = 1.0 / math.sqrt(hd)
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    assert np.all(np.isfinite(o))
    j = 123
    q[0, :] = q[0, 0]                                   # all heads share one query
    k[0, j, 0] = (q[0, 0] * 40).astype(np.float16)      # score ~ 40*|q|^2/sqrt(hd) ~ 450
    o = _run(q, k, v, pos, n_head, n_kv, hd, cap, scale, lib)
    for h in range(n_head):
        assert np.max(np.abs(o[0, h] - v[0, j, 0].astype(np.float64))) <= 1e-12


def test_stability():
    check_stability()


# ----------------------------------------------- workload generator sanity

def test_synthetic_workloads_shapes():
    w = syn.WORKLOADS["smallhead"]
    lay = syn.make_layer(w)
    assert lay["q"].shape == (1, 4, 8) and lay["q"].dtype == np.float32
    assert lay["k"].shape == (1, 64, 2, 8) and lay["k"].dtype == np.float16
    assert lay["positions"].tolist() == [63]
    again = syn.make_layer(w)
    assert np.array_equal(lay["k"], again["k"]) and np.array_equal(lay["q"], again["q"])
    r = syn.WORKLOADS["ragged"]
    assert len(r.ctx) == 32 and all(1 <= c <= 32768 for c in r.ctx)
    assert syn.WORKLOADS["7b"].kv_bytes() == 16777216
    assert syn.WORKLOADS["long"].kv_bytes() == 17203200
    assert syn.WORKLOADS["tiny"].kv_bytes() == 524288


def test_oracle_on_tiny_workload_is_finite():
    w = syn.WORKLOADS["tiny"]
    lay = syn.make_layer(w)
    o = oracle.attn_decode(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                           w.n_kv_head, w.head_dim, w.cap, w.scale, n_threads=2)
    assert o.shape == (1, 8, 128) and np.all(np.isfinite(o))
    one = oracle.attn_decode_one(lay["q"], lay["k"], lay["v"], lay["positions"], w.n_head,
                                 w.n_kv_head, w.head_dim, w.cap, w.scale, 0, 5)
    assert np.array_equal(one, o[0, 5])


def test_golden_regression_fixture():
    """The oracle still reproduces the stored fixture written by tests/golden/make_golden.py."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "smallhead_ctx16.json")
    doc = json.load(open(path))
    sh = doc["shape"]
    q = np.array([float(x) for x in doc["q_f32"]], np.float32).reshape(1, sh["n_head"], sh["head_dim"])
    kv_shape = (1, sh["cap"], sh["n_kv_head"], sh["head_dim"])
    k = np.array(doc["k_f16_bits"], np.uint16).reshape(kv_shape)
    v = np.array(doc["v_f16_bits"], np.uint16).reshape(kv_shape)
    o = oracle.attn_decode(q, k, v, np.array(doc["positions"], np.int32), sh["n_head"],
                           sh["n_kv_head"], sh["head_dim"], sh["cap"], doc["scale"])
    want = np.array([float(x) for x in doc["o_f64"]]).reshape(o.shape)
    assert np.max(np.abs(o - want)) <= 1e-15


# ------------------------------------------------------ causal multi-query

def decimal_attention_multi(q, k, v, pos, n_q, n_head, n_kv, hd, cap, scale):
    """50-digit brute force with a per-query causal limit (row t sees the first
    nkv - n_q + t + 1 rows)."""
    n_seq = q.shape[0]
    out = np.zeros((n_seq, n_q, n_head, hd))
    for s in range(n_seq):
        nkv = max(0, min(int(pos[s]) + 1, cap))
        for t in range(n_q):
            lim = nkv - n_q + t + 1
            if lim <= 0:
                continue
            sub = decimal_attention(q[s:s + 1, t], k[s:s + 1], v[s:s + 1],
                                    np.array([lim - 1], np.int32), n_head, n_kv, hd, cap, scale)
            out[s, t] = sub[0]
    return out


def check_multi_query(lib=None):
    rng = np.random.Generator(np.random.PCG64(18))
    n_q, n_head, n_kv, hd, cap = 3, 4, 2, 8, 10
    q = rng.standard_normal((2, n_q, n_head, hd), dtype=np.float32)
    k = rng.standard_normal((2, cap, n_kv, hd), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((2, cap, n_kv, hd), dtype=np.float32).astype(np.float16)
    pos = np.array([9, 1], np.int32)          # the second sequence: row 0 sees nothing
    got = oracle.attn_decode_multi(q, k, v, pos, n_q, n_head, n_kv, hd, cap, 0.4, lib=lib)
    ref = decimal_attention_multi(q, k, v, pos, n_q, n_head, n_kv, hd, cap, 0.4)
    assert np.max(np.abs(got - ref)) <= 1e-13
    assert np.all(got[1, 0] == 0)
    # one query row is the single-query oracle exactly
    one = oracle.attn_decode_multi(q[:, :1], k, v, pos, 1, n_head, n_kv, hd, cap, 0.4, lib=lib)
    single = oracle.attn_decode(q[:, 0], k, v, pos, n_head, n_kv, hd, cap, 0.4, lib=lib)
    assert np.array_equal(one[:, 0], single)


def test_multi_query_causal():
    check_multi_query()
