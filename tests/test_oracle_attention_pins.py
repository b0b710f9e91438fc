"""Pins of the oracle's decode attention (``oracle.attention``,
``oracle.decode_attention``, ``oracle.cache_kv``) to facts that do not come
from the oracle itself: closed forms (one token, a zero query, two tokens),
invariances of softmax attention (token order, a common key shift, the
scale/query trade), a saturated softmax, the grouped-query head mapping, a
50-digit evaluation with mpmath on small random cases, and the token order of
the reconstructed cache (store first, then the residual ring from its head).

The attention is the one the fused-kernel post's last section asks for
("dequant-in-SDPA": attention that reads the packed codes and expands them in
registers), i.e. softmax attention over the reconstructed fp16 cache.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import workloads as W


def _f16(a) -> np.ndarray:
    return np.asarray(a, np.float64).astype(np.float16).view(np.uint16)


def _val(u16) -> np.ndarray:
    return np.asarray(u16, np.uint16).view(np.float16).astype(np.float64)


def _rand(rng, shape, scale=1.0):
    return _f16(rng.standard_normal(shape) * scale)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    for d in (8, 64, 128):
        q, k, v = _rand(rng, (3, d)), _rand(rng, (1, d)), _rand(rng, (1, d), 5.0)
        out = O.attention(q, k, v, 1.0 / math.sqrt(d))
        assert np.array_equal(out, np.repeat(_val(v), 3, axis=0))


def test_zero_query_gives_the_mean_of_the_values():
    rng = np.random.default_rng(2)
    n, d = 37, 16
    q = np.zeros((2, d), np.uint16)
    k, v = _rand(rng, (n, d)), _rand(rng, (n, d))
    out = O.attention(q, k, v, 0.125)
    want = np.array([math.fsum(_val(v)[:, c]) / n for c in range(d)])
    np.testing.assert_allclose(out[0], want, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out[1], want, rtol=1e-14, atol=1e-15)


def test_two_tokens_follow_the_logistic_function():
    rng = np.random.default_rng(3)
    for _ in range(20):
        d = 32
        q, k, v = _rand(rng, (1, d)), _rand(rng, (2, d)), _rand(rng, (2, d))
        scale = 0.25
        dots = [sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(_val(q)[0], _val(k)[t]))
                for t in range(2)]
        delta = float(scale * (dots[0] - dots[1]))
        p0 = 1.0 / (1.0 + math.exp(-delta))
        want = p0 * _val(v)[0] + (1.0 - p0) * _val(v)[1]
        np.testing.assert_allclose(O.attention(q, k, v, scale)[0], want, rtol=1e-13, atol=1e-14)


def test_token_order_does_not_matter_but_key_value_pairing_does():
    rng = np.random.default_rng(4)
    n, d = 50, 64
    q, k, v = _rand(rng, (4, d)), _rand(rng, (n, d)), _rand(rng, (n, d))
    out = O.attention(q, k, v, 0.2)
    perm = rng.permutation(n)
    np.testing.assert_allclose(O.attention(q, k[perm], v[perm], 0.2), out, rtol=1e-12,
                               atol=1e-14)
    v2 = v.copy()
    v2[[0, 1]] = v2[[1, 0]]                    # values swapped, keys left in place
    assert not np.allclose(O.attention(q, k, v2, 0.2), out, rtol=1e-6, atol=0)


def test_common_key_shift_leaves_the_output_unchanged():
    rng = np.random.default_rng(5)
    n, d = 20, 16
    k_int = rng.integers(-8, 8, (n, d))
    u = rng.integers(-4, 4, d)
    q, v = _rand(rng, (2, d)), _rand(rng, (n, d))
    a = O.attention(q, _f16(k_int), v, 0.3)
    b = O.attention(q, _f16(k_int + u), v, 0.3)   # every score moves by scale * q.u
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_scale_trades_against_the_query():
    rng = np.random.default_rng(6)
    n, d = 30, 32
    q_int = rng.integers(-6, 7, (3, d))
    k, v = _rand(rng, (n, d)), _rand(rng, (n, d))
    np.testing.assert_allclose(O.attention(_f16(2 * q_int), k, v, 0.05),
                               O.attention(_f16(q_int), k, v, 0.1), rtol=1e-14, atol=1e-15)


def test_saturated_softmax_selects_one_value_exactly():
    rng = np.random.default_rng(7)
    n, d = 9, 8
    k = _rand(rng, (n, d), 0.01)
    k[4] = _f16(np.full(d, 100.0))
    q = _f16(np.full((1, d), 10.0))
    v = _rand(rng, (n, d))
    # score gap >= 8 * 10 * (100 - 0.05) > 7900: every other weight underflows to 0
    out = O.attention(q, k, v, 1.0)
    assert np.array_equal(out[0], _val(v)[4])


def test_grouped_query_heads_share_consecutive_kv_heads():
    rng = np.random.default_rng(8)
    batch, h_kv, r, n, d = 2, 3, 4, 11, 16
    q = _rand(rng, (batch, h_kv * r, d))
    k, v = _rand(rng, (batch * h_kv, n, d)), _rand(rng, (batch * h_kv, n, d))
    out = O.decode_attention(q, k, v, 0.25)
    for b in range(batch):
        for h in range(h_kv * r):
            j = b * h_kv + h // r
            assert np.array_equal(out[b, h], O.attention(q[b, h:h + 1], k[j], v[j], 0.25)[0])


def test_against_fifty_digit_evaluation():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(9)
    for n, d, scl in [(5, 8, 3.0), (17, 16, 1.0), (33, 24, 0.5)]:
        q, k, v = _rand(rng, (2, d), scl), _rand(rng, (n, d), scl), _rand(rng, (n, d))
        scale = 1.0 / math.sqrt(d)
        qf, kf, vf = _val(q), _val(k), _val(v)
        out = O.attention(q, k, v, scale)
        for h in range(2):
            s = [mp.mpf(scale) * mp.fsum(mp.mpf(float(qf[h, c])) * mp.mpf(float(kf[t, c]))
                                         for c in range(d)) for t in range(n)]
            m = max(s)
            e = [mp.e ** (x - m) for x in s]
            den = mp.fsum(e)
            for c in range(d):
                want = mp.fsum(e[t] / den * mp.mpf(float(vf[t, c])) for t in range(n))
                assert abs(out[h, c] - float(want)) <= 1e-14 * (1 + abs(float(want)))


def test_cache_kv_is_store_then_ring_in_token_order():
    w = W.custom(seed=12, batch=1, kv_heads=2, seq=160, head_dim=32)
    k_all, v_all = W.generate(w, 0, "k"), W.generate(w, 0, "v")
    group, bits, residual, r_cap = 32, 4, 32, 96
    st = O.Store(2, 32, 160, group, bits)
    k_ring = np.zeros((2, r_cap, 32), np.uint16)
    v_ring = np.zeros((2, r_cap, 32), np.uint16)
    s_q = head = n_res = pos = 0
    for n_new in (70, 26, 40, 24):
        rows = (head + n_res + np.arange(n_new)) % r_cap
        k_ring[:, rows] = k_all[:, pos:pos + n_new]
        v_ring[:, rows] = v_all[:, pos:pos + n_new]
        n_res += n_new
        pos += n_new
        _, s_q, head, n_res = O.flush(k_ring, v_ring, st, residual, s_q, head, n_res)
    assert s_q + n_res == 160 and head != 0 and s_q > 0
    k, v = O.cache_kv(st, s_q, k_ring, v_ring, head, n_res)
    # the residual part is the newest tokens verbatim
    assert np.array_equal(k[:, s_q:], k_all[:, s_q:]) and np.array_equal(v[:, s_q:], v_all[:, s_q:])
    # the store part is the reconstruction of the oldest tokens
    kc, ks, kz = O.quantize_keys(np.ascontiguousarray(k_all[:, :s_q]), group, bits)
    vc, vs, vz = O.quantize_values(np.ascontiguousarray(v_all[:, :s_q]), group, bits)
    assert np.array_equal(k[:, :s_q], O.dequantize_keys(kc, ks, kz, s_q, group, bits))
    assert np.array_equal(v[:, :s_q], O.dequantize_values(vc, vs, vz, group, bits))
