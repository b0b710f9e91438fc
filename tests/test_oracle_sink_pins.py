"""Pins of the oracle's KIVI-Sink functions (``sink_scores``, ``SinkState``,
``flush_sink``, ``sink_restore``) to facts that do not come from the oracle.

The method (VeloxQuant-MLX project description, section "KVSink-adapted sink
protection"): tokens with anomalously high key L2-norm (mean over the KV
heads, a running top-k of token positions) are kept fp16 and excluded from
the quantization-parameter calibration; with no sink tokens the method is
plain KIVI bit for bit; protecting planted sinks lowers the neighbours'
reconstruction error.  Each of these statements is a pin below, together with
closed-form norms, a brute-force ranking, the exclusion rule written out with
numpy and the degenerate all-sink group.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle as O
import workloads as W


def _f16(a) -> np.ndarray:
    return np.asarray(a, np.float64).astype(np.float16).view(np.uint16)


def _val(u16) -> np.ndarray:
    return np.asarray(u16, np.uint16).view(np.float16).astype(np.float64)


def test_scores_closed_forms():
    batch, heads, n, d = 2, 2, 3, 16
    k = np.zeros((batch * heads, n, d))
    k[0, 0, :2] = [3, 4]          # norm 5
    k[1, 0, 5] = -12              # norm 12  -> mean 8.5
    k[0, 1, :] = 1.0              # norm 4 (sqrt 16)
    k[1, 1, :4] = 2.0             # norm 4   -> mean 4
    k[2, 2, 7] = 0.5              # norm 0.5 -> mean 0.25 with a zero head
    s = O.sink_scores(_f16(k), heads)
    assert s.dtype == np.float32
    assert s[0, 0] == 8.5 and s[0, 1] == 4.0 and s[0, 2] == 0.0
    assert s[1, 2] == 0.25 and s[1, 0] == 0.0


def test_scores_match_float64_norms():
    rng = np.random.default_rng(1)
    batch, heads, n, d = 3, 4, 50, 128
    k = _f16(rng.standard_normal((batch * heads, n, d)) * rng.uniform(0.1, 5, (batch * heads, n, 1)))
    s = O.sink_scores(k, heads)
    ref = np.linalg.norm(_val(k), axis=2).reshape(batch, heads, n).mean(axis=1)
    np.testing.assert_allclose(s, ref, rtol=2e-6)


def test_topk_is_the_brute_force_ranking_and_merges_incrementally():
    rng = np.random.default_rng(2)
    batch, n, k_top = 3, 300, 7
    scores = rng.integers(0, 40, (batch, n)).astype(np.float32)   # many ties
    one = O.SinkState(batch, 1, 8, k_top, 16)
    one.update(scores, 0)
    inc = O.SinkState(batch, 1, 8, k_top, 16)
    for p0 in range(0, n, 37):
        inc.update(scores[:, p0:p0 + 37], p0)
    for b in range(batch):
        order = sorted(range(n), key=lambda t: (-scores[b, t], t))[:k_top]
        assert list(one.top_pos[b, :k_top]) == order
        assert list(inc.top_pos[b, :k_top]) == order
        assert one.top_count[b] == k_top


def _flush_all(k, v, group, bits, residual, state, store):
    """One flush of a whole prompt held in the ring."""
    bh, s, d = k.shape
    return O.flush_sink(k, v, store, residual, 0, 0, s, state) if state is not None else \
        O.flush(k, v, store, residual, 0, 0, s)


def test_no_sink_tokens_is_plain_kivi_bit_for_bit():
    w = W.custom(seed=3, batch=2, kv_heads=2, seq=160, head_dim=64)
    k, v = W.generate(w, 0, "k"), W.generate(w, 0, "v")
    for k_top in (0, 5):
        a = O.Store(4, 64, 160, 32, 2)
        b = O.Store(4, 64, 160, 32, 2)
        st = O.SinkState(2, 2, 64, k_top, 8)
        if k_top:                      # a top set none of whose positions is flushed
            st.top_pos[:, :k_top] = 1000 + np.arange(k_top)
            st.top_count[:] = k_top
        assert _flush_all(k, v, 32, 2, 32, None, a) == _flush_all(k, v, 32, 2, 32, st, b)
        for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero"):
            assert np.array_equal(getattr(a, name).view(np.uint32), getattr(b, name).view(np.uint32))
        assert not st.sink_count.any()


def planted(seed=4, batch=2, heads=2, s=256, d=64, sinks=((0, [3, 70, 130]), (1, [0, 200]))):
    w = W.custom(seed=seed, batch=batch, kv_heads=heads, seq=s, head_dim=d)
    k = _val(W.generate(w, 0, "k"))
    v = _val(W.generate(w, 0, "v"))
    for b, ts in sinks:
        for t in ts:
            k[b * heads:(b + 1) * heads, t] *= 40.0     # anomalously high key norm
            v[b * heads:(b + 1) * heads, t] *= 10.0
    return _f16(k), _f16(v)


def test_planted_sinks_are_selected_excluded_and_restored():
    batch, heads, s, d, group, bits, residual = 2, 2, 256, 64, 32, 2, 32
    k, v = planted()
    st = O.SinkState(batch, heads, d, 3, 8)
    st.update(O.sink_scores(k, heads), 0)
    assert set(st.top_pos[0, :3]) == {3, 70, 130}
    assert set(st.top_pos[1, :2]) == {0, 200}
    store = O.Store(batch * heads, d, s, group, bits)
    n, s_q, _, _ = O.flush_sink(k, v, store, residual, 0, 0, s, st)
    assert n == s_q == s - residual
    sinks = {b: [t for t in st.top_pos[b, :st.top_count[b]] if t < n] for b in range(batch)}
    assert list(st.sink_count) == [len(sinks[0]), len(sinks[1])]
    kf, vf = _val(k), _val(v)
    for bb in range(batch * heads):
        b = bb // heads
        excl = set(sinks[b])
        for j in range(n // group):
            toks = [t for t in range(j * group, (j + 1) * group) if t not in excl]
            for c in range(0, d, 7):
                vals = kf[bb, toks, c]
                assert store.k_zero[bb, j, c] == np.float32(vals.min() + 0.0)
                want = np.float32(np.float32(vals.max() + 0.0) - np.float32(vals.min() + 0.0)) / np.float32(3)
                assert store.k_scale[bb, j, c] == np.float32(want)
        for t in sinks[b]:
            assert not store.v_codes[bb, t].any() and not store.v_scale[bb, t].any()
            w_ = 32 // bits
            words = store.k_codes[bb, t // w_, :]
            assert not ((words >> ((t % w_) * bits)) & 3).any()   # key code slots 0
    # restored reconstruction: sinks exact, everything else as dequantized
    ky = O.dequantize_keys(store.k_codes[:, :n // 16], store.k_scale[:, :n // group],
                           store.k_zero[:, :n // group], n, group, bits)
    vy = O.dequantize_values(store.v_codes[:, :n], store.v_scale[:, :n], store.v_zero[:, :n],
                             group, bits)
    ky0, vy0 = ky.copy(), vy.copy()
    O.sink_restore(ky, vy, st)
    for bb in range(batch * heads):
        b = bb // heads
        for t in range(n):
            if t in sinks[b]:
                assert np.array_equal(ky[bb, t], k[bb, t]) and np.array_equal(vy[bb, t], v[bb, t])
            else:
                assert np.array_equal(ky[bb, t], ky0[bb, t])


def test_protection_lowers_the_neighbours_error():
    """The project description's claim: with planted high-norm sinks, the
    sink-protected cache reconstructs the other tokens better than plain KIVI."""
    batch, heads, s, d, group, bits, residual = 2, 2, 256, 64, 32, 2, 32
    k, v = planted(seed=8)
    n = s - residual
    plain = O.Store(batch * heads, d, s, group, bits)
    O.flush(k, v, plain, residual, 0, 0, s)
    st = O.SinkState(batch, heads, d, 3, 8)
    st.update(O.sink_scores(k, heads), 0)
    prot = O.Store(batch * heads, d, s, group, bits)
    O.flush_sink(k, v, prot, residual, 0, 0, s, st)
    sinks = {b: set(int(t) for t in st.top_pos[b, :st.top_count[b]] if t < n) for b in range(batch)}
    mask = np.ones((batch * heads, n), bool)
    for bb in range(batch * heads):
        for t in sinks[bb // heads]:
            mask[bb, t] = False

    def key_err(store):
        y = _val(O.dequantize_keys(store.k_codes[:, :n // 16], store.k_scale[:, :n // group],
                                   store.k_zero[:, :n // group], n, group, bits))
        return float(((y - _val(k)[:, :n]) ** 2)[mask].mean())
    assert key_err(prot) < 0.5 * key_err(plain)


def test_all_sink_group_and_sink_store_capacity():
    batch, heads, d, group, bits = 1, 1, 32, 32, 4
    k = _f16(np.random.default_rng(5).standard_normal((1, 64, d)))
    v = k.copy()
    st = O.SinkState(batch, heads, d, 32, 32)
    st.top_pos[0, :32] = np.arange(32)             # the whole first group
    st.top_count[0] = 32
    store = O.Store(1, d, 64, group, bits)
    n, _, _, _ = O.flush_sink(k, v, store, 0, 0, 0, 64, st)
    assert n == 64
    assert not store.k_scale[0, 0].any() and not store.k_zero[0, 0].any()
    assert not store.k_codes[0, :4].any()          # 32 tokens x 4 bits = 4 word rows
    assert store.k_scale[0, 1].all()
    small = O.SinkState(batch, heads, d, 32, 31)   # 32 sinks do not fit
    small.top_pos[0, :32] = np.arange(32)
    small.top_count[0] = 32
    with pytest.raises(ValueError):
        O.flush_sink(k, v, O.Store(1, d, 64, group, bits), 0, 0, 0, 64, small)
    assert small.sink_count[0] == 0
