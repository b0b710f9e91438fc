"""KIVI-Sink on the GPU (``kivi_sink_update``, ``kivi_flush_sink``,
``kivi_sink_restore``) against the oracle, bit for bit: the binary32 scores
and the ranked top-k, the sink-protected store, the sink store and the
restored reconstruction, over prefill and decode sequences with ring
wrap-around, planted high-norm tokens, every code width and two head dims."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_same, bits32, host_f32_bits, host_u16, host_u32, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_cache_quantization_kivi_gb300 as K  # noqa: E402


class SinkPair:
    """A GPU cache + sinks and the oracle's mirror, fed the same tokens."""

    def __init__(self, layers, batch, heads, d, bits, group, residual, r_cap, cap, k_top,
                 sink_cap, seed, plant_every=0):
        self.layers, self.batch, self.heads, self.d = layers, batch, heads, d
        self.bh = batch * heads
        self.group, self.bits, self.residual, self.r_cap, self.cap = group, bits, residual, r_cap, cap
        self.cache = K.KiviCache(layers, self.bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                                 residual=residual)
        self.sinks = K.KiviSinks(self.cache, batch, k_top, sink_cap)
        self.w = W.custom(seed=seed, batch=batch, kv_heads=heads, seq=cap + r_cap, head_dim=d)
        self.plant_every = plant_every
        self.ring_k = [np.zeros((self.bh, r_cap, d), np.uint16) for _ in range(layers)]
        self.ring_v = [np.zeros((self.bh, r_cap, d), np.uint16) for _ in range(layers)]
        self.stores = [O.Store(self.bh, d, cap, group, bits) for _ in range(layers)]
        self.states = [O.SinkState(batch, heads, d, k_top, sink_cap) for _ in range(layers)]
        self.s_q = self.head = self.n_res = self.pos = 0

    def tokens(self, l, kind, n):
        x = W.generate(self.w, l, kind, tok0=self.pos, n_tok=n)
        if self.plant_every:
            f = x.view(np.float16).astype(np.float32)
            rng = np.random.default_rng(self.pos * 7 + l)
            for b in range(self.batch):
                for i in range(n):
                    if rng.integers(self.plant_every) == 0:   # a high-norm token
                        f[b * self.heads:(b + 1) * self.heads, i] *= (30.0 if kind == "k" else 8.0)
            x = f.astype(np.float16).view(np.uint16)
        return np.ascontiguousarray(x)

    def append(self, n_new, flush=True):
        rows = (self.head + self.n_res + np.arange(n_new)) % self.r_cap
        i0 = self.n_res
        for l in range(self.layers):
            k, v = self.tokens(l, "k", n_new), self.tokens(l, "v", n_new)
            self.ring_k[l][:, rows] = k
            self.ring_v[l][:, rows] = v
            self.cache.append(l, to_dev(k), to_dev(v))
            self.states[l].update(O.sink_scores(k, self.heads), self.s_q + i0)
        self.cache.advance(n_new)
        self.sinks.update(i0, n_new)
        self.n_res += n_new
        self.pos += n_new
        if flush:
            n_gpu = self.sinks.flush()
            for l in range(self.layers):
                n, s_q, head, n_res = O.flush_sink(self.ring_k[l], self.ring_v[l], self.stores[l],
                                                   self.residual, self.s_q, self.head, self.n_res,
                                                   self.states[l])
            assert n_gpu == n
            self.s_q, self.head, self.n_res = s_q, head, n_res
            assert (self.cache.s_q, self.cache.res_head, self.cache.n_res) == (s_q, head, n_res)

    def check(self):
        torch.cuda.synchronize()
        assert K.kivi_device_fault() == 0
        sk = self.sinks
        for l in range(self.layers):
            st, o = self.stores[l], self.states[l]
            kt = self.sinks.k_top
            cnt = sk.top_count[l].cpu().numpy()
            assert np.array_equal(cnt, o.top_count), (l, cnt, o.top_count)
            tp = sk.top_pos[l].cpu().numpy()
            ts = host_f32_bits(sk.top_score[l])
            for b in range(self.batch):
                c = int(cnt[b])
                assert np.array_equal(tp[b, :c], o.top_pos[b, :c]), (l, b)
                assert np.array_equal(ts[b, :c], bits32(o.top_score[b, :c])), (l, b)
            assert_same("key codes", host_u32(self.cache.k_codes[l]), st.k_codes)
            assert_same("key scale", host_f32_bits(self.cache.k_scale[l]), bits32(st.k_scale))
            assert_same("key zero", host_f32_bits(self.cache.k_zero[l]), bits32(st.k_zero))
            assert_same("value codes", host_u32(self.cache.v_codes[l]), st.v_codes)
            assert_same("value scale", host_f32_bits(self.cache.v_scale[l]), bits32(st.v_scale))
            assert_same("value zero", host_f32_bits(self.cache.v_zero[l]), bits32(st.v_zero))
            scnt = sk.sink_count[l].cpu().numpy()
            assert np.array_equal(scnt, o.sink_count), (l, scnt, o.sink_count)
            spos = sk.sink_pos[l].cpu().numpy()
            for b in range(self.batch):
                c = int(scnt[b])
                assert np.array_equal(spos[b, :c], o.sink_pos[b, :c])
                for h in range(self.heads):
                    bb = b * self.heads + h
                    assert np.array_equal(host_u16(sk.sink_k[l][bb, :c]), o.sink_k[bb, :c])
                    assert np.array_equal(host_u16(sk.sink_v[l][bb, :c]), o.sink_v[bb, :c])
        # dequantized store with the sinks restored
        ky, vy = self.cache.dequantize()
        sk.restore(ky, vy)
        torch.cuda.synchronize()
        for l in range(self.layers):
            kref, vref = O.cache_kv(self.stores[l], self.s_q, self.ring_k[l], self.ring_v[l],
                                    self.head, 0)
            O.sink_restore(kref, vref, self.states[l])
            assert_same("restored keys", host_u16(ky[l]), kref)
            assert_same("restored values", host_u16(vy[l]), vref)


@pytest.mark.parametrize("bits,group,d", [(2, 32, 128), (4, 64, 128), (8, 128, 128),
                                          (2, 64, 64), (4, 32, 64), (2, 16, 128), (8, 16, 64)])
def test_sink_prefill_flush(bits, group, d):
    batch, heads, S = 2, 2, 8 * group
    pair = SinkPair(2, batch, heads, d, bits, group, group, r_cap=S, cap=S, k_top=5,
                    sink_cap=8, seed=40 + bits + group + d, plant_every=60)
    pair.append(S, flush=True)
    assert pair.s_q == S - group
    assert (pair.sinks.sink_count.cpu().numpy() > 0).all()
    pair.check()


@pytest.mark.parametrize("bits,group,r_groups", [(2, 32, 4), (4, 64, 4), (4, 16, 5)])
def test_sink_decode_sequence_with_ring_wrap(bits, group, r_groups):
    batch, heads, d = 3, 2, 128
    pair = SinkPair(2, batch, heads, d, bits, group, group, r_cap=r_groups * group, cap=16 * group,
                    k_top=6, sink_cap=40, seed=70 + bits, plant_every=90)
    pair.append(3 * group)                      # a prefill
    rng = np.random.default_rng(bits)
    while pair.s_q + pair.n_res < 14 * group:
        n = int(min(rng.integers(1, group), pair.r_cap - pair.n_res))
        pair.append(n)
    assert pair.head > 0
    pair.check()


def test_no_top_k_is_plain_kivi():
    batch, heads, d, group, bits = 2, 2, 128, 32, 2
    pair = SinkPair(1, batch, heads, d, bits, group, group, r_cap=256, cap=256, k_top=0,
                    sink_cap=0, seed=5, plant_every=40)
    pair.append(256)
    pair.check()
    st = O.Store(pair.bh, d, 256, group, bits)
    O.flush(pair.ring_k[0], pair.ring_v[0], st, group, 0, 0, 256)
    assert_same("plain key codes", host_u32(pair.cache.k_codes[0]), st.k_codes)
    assert_same("plain value codes", host_u32(pair.cache.v_codes[0]), st.v_codes)


def test_sink_store_overflow_keeps_the_earliest_sinks():
    """A flush whose sinks do not all fit the sink store records the overflow
    (bit 1 of the fault word), stores the earliest flushed sinks that fit,
    and quantizes the other flushed top-k tokens as plain tokens: store, sink
    store and restored reconstruction equal the oracle's flush over a top-k
    cut down to the sinks that fit."""
    batch, heads, d, group, bits, cap_sinks = 2, 2, 128, 32, 4, 3
    pair = SinkPair(1, batch, heads, d, bits, group, group, r_cap=256, cap=256, k_top=8,
                    sink_cap=cap_sinks, seed=9, plant_every=20)
    k = pair.tokens(0, "k", 256)
    v = pair.tokens(0, "v", 256)
    pair.ring_k[0][:] = k
    pair.ring_v[0][:] = v
    pair.cache.append(0, to_dev(k), to_dev(v))
    pair.cache.advance(256)
    full = pair.states[0]
    full.update(O.sink_scores(k, heads), 0)
    pair.sinks.update(0, 256)
    n = pair.sinks.flush()
    torch.cuda.synchronize()
    assert K.kivi_device_fault() == 2
    assert (pair.sinks.sink_count[0].cpu().numpy() == cap_sinks).all()
    # the oracle refuses an overflowing flush; its expectation is the flush
    # over the top-k cut down to the earliest flushed positions that fit
    cut = O.SinkState(batch, heads, d, 8, cap_sinks)
    excess = []
    for b in range(batch):
        flushed = sorted(int(p) for p in full.top_pos[b, :full.top_count[b]] if p < n)
        assert len(flushed) > cap_sinks, flushed     # every sequence overflows
        cut.top_pos[b, :cap_sinks] = flushed[:cap_sinks]
        cut.top_count[b] = cap_sinks
        excess += [(b, p) for p in flushed[cap_sinks:]]
    n_o, s_q, head, n_res = O.flush_sink(pair.ring_k[0], pair.ring_v[0], pair.stores[0], group,
                                         0, 0, 256, cut)
    assert n_o == n
    pair.s_q, pair.head, pair.n_res = s_q, head, n_res
    # the running top-k itself is untouched by the flush
    cut.top_pos[:], cut.top_score[:], cut.top_count[:] = (full.top_pos, full.top_score,
                                                           full.top_count)
    pair.states[0] = cut
    pair.check()
    # the excess top-k tokens kept their values: quantized rows, not zeroed ones
    vs = pair.cache.v_scale[0].cpu().numpy()
    for b, p in excess:
        assert (vs[b * heads:(b + 1) * heads, p] > 0).all(), (b, p)


def attention_bound_check(q16, k, v, got, sm_scale, batch):
    """Every output element within (2^-16 + 2^-16 A) B of the oracle's
    attention (the bound of tests/test_gpu_attention.py)."""
    ref = O.decode_attention(q16.view(np.uint16), k, v, sm_scale)
    kf = k.view(np.float16).astype(np.float64)
    vf = v.view(np.float16).astype(np.float64)
    qf = q16.astype(np.float64)
    h_q = q16.shape[1]
    h_kv = k.shape[0] // batch
    r = h_q // h_kv
    for b in range(batch):
        for h in range(h_q):
            j = b * h_kv + h // r
            sc = sm_scale * (kf[j] @ qf[b, h])
            p = np.exp(sc - sc.max())
            p /= p.sum()
            A = sm_scale * np.max(np.abs(kf[j]) @ np.abs(qf[b, h]))
            B = p @ np.abs(vf[j])
            tol = (2.0 ** -16) * (1.0 + A) * B + 1e-30
            assert (np.abs(got[b, h] - ref[b, h]) <= tol).all(), (b, h)
    return ref


@pytest.mark.parametrize("bits,group,d", [(2, 32, 128), (4, 64, 128), (8, 16, 128), (2, 16, 64),
                                          (4, 32, 256)])
def test_attention_over_sink_protected_cache(bits, group, d):
    """Decode attention over a sink-protected cache equals the oracle's
    attention over the restored cache (store dequantized, sinks' fp16 rows
    put back, residual appended), within the attention bound; without the
    sink store the stored sinks' zeroed slots would be attended instead."""
    batch, heads = 2, 2
    pair = SinkPair(2, batch, heads, d, bits, group, group, r_cap=4 * group, cap=16 * group,
                    k_top=6, sink_cap=40, seed=90 + bits + group, plant_every=50)
    pair.append(3 * group)
    rng = np.random.default_rng(bits + group)
    while pair.s_q + pair.n_res < 11 * group:
        pair.append(int(min(rng.integers(1, group), pair.r_cap - pair.n_res)))
    assert (pair.sinks.sink_count.cpu().numpy() > 0).all() and pair.n_res > 0
    h_q = 4 * heads
    q16 = (rng.standard_normal((2, batch, h_q, d)) * 0.5).astype(np.float16)
    qd = torch.from_numpy(q16.view(np.int16)).view(torch.float16).cuda()
    sc = 1.0 / np.sqrt(d)
    differs = False
    for n_split in (1, 3):
        got = pair.cache.decode_attention(qd, batch, sm_scale=sc, n_split=n_split,
                                          sinks=pair.sinks).cpu().numpy().astype(np.float64)
        plain = pair.cache.decode_attention(qd, batch, sm_scale=sc,
                                            n_split=n_split).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        assert K.kivi_device_fault() == 0
        for l in range(2):
            k, v = O.cache_kv(pair.stores[l], pair.s_q, pair.ring_k[l], pair.ring_v[l],
                              pair.head, pair.n_res)
            O.sink_restore(k, v, pair.states[l])
            ref = attention_bound_check(q16[l], k, v, got[l], sc, batch)
            differs |= bool(np.abs(plain[l] - ref).max() > 1e-3)
    assert differs


@pytest.mark.parametrize("batch,heads,d", [(2, 1, 128), (1, 3, 128), (3, 5, 64), (2, 8, 128),
                                           (1, 11, 96), (2, 9, 256), (1, 64, 64), (1, 65, 32),
                                           (1, 300, 32)])
def test_sink_scores_every_head_count(batch, heads, d):
    """The scores scratch equals the oracle's scores bit for bit for head
    counts below, at and above the eight warps of a score block (each warp
    takes heads w, w + 8, ...), head dims that stage in one, one and a half
    (96) and four 64-channel passes, a token count with a ragged last tile,
    and more than 64 heads (the thread-per-token kernel); then the whole
    sink pipeline on those tokens."""
    group = 32
    pair = SinkPair(2, batch, heads, d, 2, group, group, r_cap=4 * group, cap=8 * group,
                    k_top=5, sink_cap=12, seed=heads * 10 + batch, plant_every=9)
    n = 3 * group + 7
    pair.append(n, flush=False)
    torch.cuda.synchronize()
    for l in range(pair.layers):
        want = O.sink_scores(pair.ring_k[l][:, :n], heads)
        got = host_f32_bits(pair.sinks.scores[l])[:, :n]
        assert np.array_equal(got, bits32(want)), (l, heads)
    pair.append(group - 10)     # 125 of 128 ring rows, then a flush of 64
    pair.check()


@pytest.mark.slow
def test_sink_prefill_full_size_as_benchmarked():
    """The benchmark's KIVI-Sink step (llama3_2_3b_prefill: 28 layers x 8 KV
    heads x 4096 tokens, top 5 per sequence) in its own launch configuration;
    two layers are compared with the oracle in full: the ranked top-k, the
    sink-protected store, the sink store and the restored reconstruction."""
    import importlib.util
    import os
    spec = importlib.util.spec_from_file_location(
        "bench_mod", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                  "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dev = torch.device("cuda", 0)
    wl = bench.make_workload("llama3_2_3b_prefill", dev, sink=True)
    stream = torch.cuda.current_stream(dev)
    wl.step(stream)
    wl.step(stream)                       # a second step from the reset state
    torch.cuda.synchronize()
    assert K.kivi_device_fault() == 0
    w, c, sk = wl.w, wl.cache, wl.sinks
    heads = w.bh // w.batch
    for l in (0, w.layers - 1):
        k = np.ascontiguousarray(wl.k_host[l])
        v = np.ascontiguousarray(wl.v_host[l])
        st = O.SinkState(w.batch, heads, w.head_dim, wl.K_TOP, 2 * wl.K_TOP)
        st.update(O.sink_scores(k, heads), 0)
        store = O.Store(w.bh, w.head_dim, w.seq, w.group, w.bits)
        n, s_q, _, _ = O.flush_sink(k, v, store, w.residual, 0, 0, w.seq, st)
        assert n == s_q == wl.n
        cnt = sk.top_count[l].cpu().numpy()
        assert np.array_equal(cnt, st.top_count)
        assert np.array_equal(sk.top_pos[l].cpu().numpy()[:, :wl.K_TOP], st.top_pos[:, :wl.K_TOP])
        assert_same("key codes", host_u32(c.k_codes[l]), store.k_codes)
        assert_same("key scale", host_f32_bits(c.k_scale[l]), bits32(store.k_scale))
        assert_same("key zero", host_f32_bits(c.k_zero[l]), bits32(store.k_zero))
        assert_same("value codes", host_u32(c.v_codes[l]), store.v_codes)
        assert_same("value scale", host_f32_bits(c.v_scale[l]), bits32(store.v_scale))
        assert np.array_equal(sk.sink_count[l].cpu().numpy(), st.sink_count)
        for b in range(w.batch):
            m = int(st.sink_count[b])
            assert m > 0
            assert np.array_equal(sk.sink_pos[l].cpu().numpy()[b, :m], st.sink_pos[b, :m])
        kref, vref = O.cache_kv(store, n, k, v, 0, 0)
        O.sink_restore(kref, vref, st)
        assert_same("restored keys", host_u16(wl.k_out[l]), kref)
        assert_same("restored values", host_u16(wl.v_out[l]), vref)


class TiedPair(SinkPair):
    """Key rows copied: in each sequence the tokens at `ties[b]` get the same
    high-norm key row in every head, so their scores are equal bit for bit
    and the ranking falls to the positions."""

    def __init__(self, *args, ties, **kw):
        super().__init__(*args, **kw)
        self.ties = ties

    def tokens(self, l, kind, n):
        x = super().tokens(l, kind, n)
        if kind == "k":
            f = x.view(np.float16).astype(np.float32)
            for b, pos in enumerate(self.ties):
                hs = slice(b * self.heads, (b + 1) * self.heads)
                row = f[hs, pos[0] - self.pos] * 20.0
                for t in pos:
                    f[hs, t - self.pos] = row
            x = np.ascontiguousarray(f.astype(np.float16).view(np.uint16))
        return x


def test_sink_top_k_ties_across_and_within_tiles():
    """Seven tokens with the same score and k = 5: the five earliest win.
    Sequence 0 spreads them over three 32-token score tiles (two, three and
    two of them), sequence 1 puts all seven in one tile, sequence 2 puts one
    in each of seven tiles; the ranked top-k and everything after it equal
    the oracle's."""
    ties = [(5, 6, 33, 40, 63, 100, 127), (64, 65, 66, 67, 68, 69, 70),
            (3, 35, 67, 99, 131, 163, 195)]
    pair = TiedPair(2, len(ties), 2, 128, 2, 32, 32, r_cap=256, cap=256, k_top=5, sink_cap=8,
                    seed=31, ties=ties)
    pair.append(256)
    for l in range(pair.layers):
        tp = pair.sinks.top_pos[l].cpu().numpy()
        for b, pos in enumerate(ties):
            assert list(tp[b, :5]) == list(pos[:5]), (l, b, tp[b])
    pair.check()


@pytest.mark.parametrize("k_top,plant_every", [(8, 6), (20, 10), (64, 4)])
def test_sink_many_tiles_dense_candidates(k_top, plant_every):
    """Many high-norm tokens (one in `plant_every`) over 16 score tiles per
    sequence, so that most tiles hold several of the sequence's top-k: k = 8
    (the score blocks select), 20 and 64 (the select kernel); a second update
    and flush merge into the kept top-k."""
    pair = SinkPair(2, 2, 2, 128, 4, 64, 64, r_cap=512, cap=1024, k_top=k_top,
                    sink_cap=2 * k_top + 8, seed=k_top, plant_every=plant_every)
    pair.append(512)
    pair.append(448)
    pair.check()
