"""Decode attention over the packed cache (``kivi_decode_attention``) against
the binary64 oracle.

The cache is filled through the library's own flush (whose bit-exact parity
the flush tests establish) while the oracle replays the same flushes; the
expected output is the oracle's attention over ``oracle.cache_kv`` (the
dequantized store followed by the residual ring).  Floating point decides
no integer here, so the comparison uses a bound derived from the arithmetic
(binary32 with fp16 tensor-core inputs):

    |out - ref| <= (2^-16 + 2^-16 * A) * B + 1e-30       per element

with A = scale * max_t sum_c |q_c k_tc| (the largest score magnitude a rounding
error can be proportional to) and B = sum_t p_t |v_tc| (the softmax-weighted
value magnitude of that output element).  It covers the binary32 dot-product
accumulation of the scores (about 2^-19 A, doubled for the maximum), the
exp2 and probability-split errors (2^-21) and the accumulation of the
weighted values over up to a few hundred tensor-core steps (2^-17 B).
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_cache_quantization_kivi_gb300 as K  # noqa: E402

D = 128


@pytest.fixture(autouse=True, params=["mma", "tcgen05"])
def attention_kernel(request, monkeypatch):
    """Every test runs on both decode-attention kernels: the default
    register-operand one and the warp-specialised tensor-memory one that
    KIVI_ATTENTION_KERNEL=tcgen05 selects (read by the library at each call;
    it takes the calls at G >= 32, the default kernel keeps G = 16)."""
    monkeypatch.setenv("KIVI_ATTENTION_KERNEL", request.param)
    return request.param


class Pair:
    """A GPU cache and the oracle's mirror of it, filled with the same tokens."""

    def __init__(self, layers, bh, bits, group, residual, r_cap, cap, seed, kdist=None, d=D):
        self.layers, self.bh, self.bits, self.group = layers, bh, bits, group
        self.residual, self.r_cap, self.cap = residual, r_cap, cap
        self.cache = K.KiviCache(layers, bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                                 residual=residual)
        self.w = W.custom(seed=seed, batch=1, kv_heads=bh, seq=cap + r_cap, head_dim=d,
                          keys=kdist or W.Dist(W.NORMAL, 1.0, n_outliers=4, outlier_mult=15.0))
        self.ring_k = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
        self.ring_v = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
        self.stores = [O.Store(bh, d, cap, group, bits) for _ in range(layers)]
        self.s_q = self.head = self.n_res = self.pos = 0

    def append(self, n_new, flush=True):
        rows = (self.head + self.n_res + np.arange(n_new)) % self.r_cap
        for l in range(self.layers):
            k = W.generate(self.w, l, "k", tok0=self.pos, n_tok=n_new)
            v = W.generate(self.w, l, "v", tok0=self.pos, n_tok=n_new)
            self.ring_k[l][:, rows] = k
            self.ring_v[l][:, rows] = v
            self.cache.append(l, to_dev(k), to_dev(v))
        self.cache.advance(n_new)
        self.n_res += n_new
        self.pos += n_new
        if flush:
            self.cache.flush()
            for l in range(self.layers):
                _, s_q, head, n_res = O.flush(self.ring_k[l], self.ring_v[l], self.stores[l],
                                              self.residual, self.s_q, self.head, self.n_res)
            self.s_q, self.head, self.n_res = s_q, head, n_res
            assert (self.cache.s_q, self.cache.res_head, self.cache.n_res) == (s_q, head, n_res)

    def set_state(self, s_q, head, n_res):
        self.s_q, self.head, self.n_res = s_q, head, n_res
        self.cache.reset(s_q=s_q, res_head=head, n_res=n_res)

    def kv(self, l):
        return O.cache_kv(self.stores[l], self.s_q, self.ring_k[l], self.ring_v[l], self.head,
                          self.n_res)


def queries(layers, batch, h_q, seed, scale=1.0, d=D):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((layers, batch, h_q, d)) * scale).astype(np.float16)


def run_gpu(pair, q16, batch, n_split=None, sm_scale=None):
    q = torch.from_numpy(q16.view(np.int16)).view(torch.float16).cuda()
    out = pair.cache.decode_attention(q, batch, sm_scale=sm_scale, n_split=n_split)
    torch.cuda.synchronize()
    assert K.kivi_device_fault() == 0
    return out.cpu().numpy().astype(np.float64)


def check(pair, q16, batch, got, sm_scale):
    """Compare every output element with the oracle under the derived bound."""
    h_q = q16.shape[2]
    h_kv = pair.bh // batch
    r = h_q // h_kv
    worst = 0.0
    for l in range(pair.layers):
        k, v = pair.kv(l)
        ref = O.decode_attention(q16[l].view(np.uint16), k, v, sm_scale)
        kf = k.view(np.float16).astype(np.float64)
        vf = v.view(np.float16).astype(np.float64)
        qf = q16[l].astype(np.float64)
        for b in range(batch):
            for h in range(h_q):
                j = b * h_kv + h // r
                s = sm_scale * (kf[j] @ qf[b, h])
                p = np.exp(s - s.max())
                p /= p.sum()
                A = sm_scale * np.max(np.abs(kf[j]) @ np.abs(qf[b, h]))
                B = p @ np.abs(vf[j])
                tol = (2.0 ** -16) * (1.0 + A) * B + 1e-30
                err = np.abs(got[l, b, h] - ref[b, h])
                bad = err > tol
                assert not bad.any(), (f"layer {l} seq {b} head {h}: {bad.sum()} channels off; "
                                       f"max err {err.max():.3e}, tol at worst "
                                       f"{tol[np.argmax(err / tol)]:.3e}")
                worst = max(worst, float((err / tol).max()))
    return worst


COMBOS = [(b, g) for b in (2, 4, 8) for g in (16, 32, 64, 128)]


@pytest.mark.parametrize("bits,group", COMBOS)
def test_attention_store_and_residual(bits, group):
    batch, h_kv, r = 2, 2, 4
    pair = Pair(1, batch * h_kv, bits, group, residual=group, r_cap=4 * group, cap=8 * group,
                seed=300 + bits + group)
    for n in (3 * group // 2, group + 5, 2 * group - 3, group + 11):
        pair.append(n)
    assert pair.s_q > 0 and pair.n_res > 0
    q = queries(1, batch, h_kv * r, 7)
    sc = 1.0 / math.sqrt(D)
    for n_split in (1, 2, 3):
        check(pair, q, batch, run_gpu(pair, q, batch, n_split=n_split, sm_scale=sc), sc)


@pytest.mark.parametrize("d,bits,group", [(64, 2, 16), (64, 2, 32), (64, 4, 64), (64, 8, 32),
                                          (64, 8, 16), (256, 2, 16), (256, 2, 32), (256, 4, 64),
                                          (256, 2, 128), (256, 8, 128), (256, 8, 16)])
def test_attention_head_dims(d, bits, group):
    """head_dim 64 and 256 (each width, G = 16 with its half-tile store end,
    the shared 2-bit key tables at G >= 32, and at 256 / 8 bits / G = 16 the
    one-stage ring): store and residual under 1 to 3 splits, as at 128."""
    batch, h_kv, r = 2, 2, 4
    pair = Pair(1, batch * h_kv, bits, group, residual=group, r_cap=4 * group, cap=8 * group,
                seed=700 + d + bits + group, d=d)
    for n in (3 * group // 2, group + 5, 2 * group - 3, group + 11):
        pair.append(n)
    assert pair.s_q > 0 and pair.n_res > 0
    q = queries(1, batch, h_kv * r, 17, d=d)
    sc = 1.0 / math.sqrt(d)
    for n_split in (1, 2, 3):
        check(pair, q, batch, run_gpu(pair, q, batch, n_split=n_split, sm_scale=sc), sc)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_attention_g16_store_ending_mid_tile(bits):
    """G = 16 lets the store end half way through a 32-token tile (here at
    240 tokens, 16 short of the capacity, after flushes of 16 to 48 tokens
    through an 80-row ring): that tile's first 16 tokens are attended and the
    rest of the tile is not read.  Uniform weights (q = 0) make a dropped or
    an extra (zero) token visible."""
    batch, h_kv, r = 2, 2, 2
    pair = Pair(2, batch * h_kv, bits, 16, residual=16, r_cap=80, cap=256, seed=80 + bits)
    for n in (50, 30, 17, 40, 29, 45, 21, 33):
        pair.append(n)
    assert (pair.s_q, pair.n_res, pair.head) == (240, 25, 0)
    sc = 1.0 / math.sqrt(D)
    q = queries(2, batch, h_kv * r, 31 + bits)
    for n_split in (1, 2, 5):
        check(pair, q, batch, run_gpu(pair, q, batch, n_split=n_split, sm_scale=sc), sc)
    q0 = np.zeros_like(q)
    assert check(pair, q0, batch, run_gpu(pair, q0, batch, n_split=3, sm_scale=1.0), 1.0) < 1.0
    pair.set_state(pair.s_q, pair.head, 0)            # store only, ending mid-tile
    check(pair, q, batch, run_gpu(pair, q, batch, n_split=4, sm_scale=sc), sc)


@pytest.mark.parametrize("r", [1, 2, 8])
def test_attention_gqa_ratios_and_layers(r):
    batch, h_kv, layers = 3, 2, 3
    pair = Pair(layers, batch * h_kv, 2, 32, residual=32, r_cap=128, cap=512, seed=40 + r)
    for n in (100, 70, 80, 33):
        pair.append(n)
    q = queries(layers, batch, h_kv * r, 11 + r)
    sc = 1.0 / math.sqrt(D)
    check(pair, q, batch, run_gpu(pair, q, batch, sm_scale=sc), sc)


def test_attention_residual_only_store_only_and_single_token():
    batch, h_kv, r = 1, 2, 4
    sc = 0.09
    pair = Pair(1, batch * h_kv, 4, 64, residual=64, r_cap=128, cap=256, seed=5)
    pair.append(37, flush=False)                     # residual only, ragged tile
    q = queries(1, batch, h_kv * r, 3)
    check(pair, q, batch, run_gpu(pair, q, batch, sm_scale=sc), sc)
    pair.append(91, flush=True)                      # now a store too
    assert pair.s_q == 64
    s_q, head = pair.s_q, pair.head
    pair.set_state(s_q, head, 0)                     # store only
    check(pair, q, batch, run_gpu(pair, q, batch, n_split=2, sm_scale=sc), sc)
    pair.set_state(0, head, 1)                       # a single residual token
    out = run_gpu(pair, q, batch, sm_scale=sc)
    check(pair, q, batch, out, sc)


def test_attention_ring_wraps_and_many_splits():
    batch, h_kv, r = 2, 1, 4
    pair = Pair(2, batch * h_kv, 2, 32, residual=32, r_cap=96, cap=1024, seed=9)
    wrapped = False
    for n in [40] * 22:
        pair.append(n)
        wrapped |= pair.head + pair.n_res > 96
    assert wrapped and pair.s_q > 700
    q = queries(2, batch, h_kv * r, 21)
    sc = 1.0 / math.sqrt(D)
    outs = [run_gpu(pair, q, batch, n_split=s, sm_scale=sc) for s in (1, 4, 7, 26)]
    for o in outs:
        check(pair, q, batch, o, sc)


def test_attention_uniform_weights_expose_every_token():
    """q = 0 gives every token the same weight: the output is the plain mean
    of the values, so one missing or duplicated token shifts it by ~|v|/n."""
    batch, h_kv, r = 1, 2, 2
    pair = Pair(1, batch * h_kv, 8, 32, residual=32, r_cap=128, cap=512, seed=13)
    for n in (96, 64, 80, 70):
        pair.append(n)
    q = np.zeros((1, batch, h_kv * r, D), np.float16)
    got = run_gpu(pair, q, batch, n_split=3, sm_scale=1.0)
    worst = check(pair, q, batch, got, 1.0)
    assert worst < 1.0
    k, v = pair.kv(0)
    mean = v.view(np.float16).astype(np.float64).mean(axis=1)     # [bh, D]
    np.testing.assert_allclose(got[0, 0, :2], np.repeat(mean[0:1], 2, 0), rtol=2e-5, atol=1e-6)


def test_attention_saturated_softmax():
    batch, h_kv, r = 1, 1, 4
    pair = Pair(1, 1, 4, 32, residual=32, r_cap=128, cap=256, seed=17)
    for n in (80, 80, 40):
        pair.append(n)
    q = queries(1, batch, h_kv * r, 5, scale=30.0)      # scores in the hundreds
    check(pair, q, batch, run_gpu(pair, q, batch, sm_scale=0.5), 0.5)


def test_attention_rejects_bad_arguments():
    pair = Pair(1, 2, 2, 32, residual=32, r_cap=64, cap=128, seed=1)
    pair.append(64)
    c = pair.cache
    q = torch.zeros((1, 2, 8, D), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 2, 8, D), dtype=torch.float32, device="cuda")
    with pytest.raises(K.KiviError):
        K.kivi_decode_attention(c.layers, 1, c.state, 3, 8, 0.1, [q[0]], [out[0]])  # bh % batch
    with pytest.raises(K.KiviError):
        K.kivi_decode_attention(c.layers, 1, c.state, 2, 9, 0.1, [q[0]], [out[0]])  # r = 9
    with pytest.raises(K.KiviError):
        K.kivi_decode_attention(c.layers, 1, c.state, 1, 18, 0.1, [q[0]], [out[0]])  # r > 8
    with pytest.raises(K.KiviError):
        K.kivi_decode_attention(c.layers, 1, c.state, 2, 8, 0.1, [q[0]], [out[0]], n_split=2)
    c96 = K.KiviCache(1, 2, 96, r_cap=64, cap=128, group=32, bits=2, residual=32)
    q96 = torch.zeros((2, 8, 96), dtype=torch.float16, device="cuda")
    o96 = torch.zeros((2, 8, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(K.KiviError):                                     # head_dim 96
        K.kivi_decode_attention(c96.layers, 1, c96.state, 2, 8, 0.1, [q96], [o96])
    torch.cuda.synchronize()
    assert not out.any() and not o96.any()


def fill_decode_store(w, cache, r_cap):
    """Every layer's store quantized from the workload's first store_prefill
    tokens (full-tensor calls), the rings holding the next r_cap tokens."""
    n = w.store_prefill
    for l in range(w.layers):
        k = to_dev(W.generate(w, l, "k", n_tok=n))
        v = to_dev(W.generate(w, l, "v", n_tok=n))
        K.kivi_quantize_keys(k, w.group, w.bits, cache.k_codes[l][:, :n * w.bits // 32],
                             cache.k_scale[l][:, :n // w.group], cache.k_zero[l][:, :n // w.group])
        K.kivi_quantize_values(v, w.group, w.bits, cache.v_codes[l][:, :n],
                               cache.v_scale[l][:, :n], cache.v_zero[l][:, :n])
        cache.k_res[l].copy_(to_dev(W.generate(w, l, "k", tok0=n, n_tok=r_cap)))
        cache.v_res[l].copy_(to_dev(W.generate(w, l, "v", tok0=n, n_tok=r_cap)))
        del k, v
    cache.reset(s_q=n, res_head=0, n_res=r_cap)


@pytest.mark.slow
def test_attention_batched_decode_full_size_sampled():
    """The decode workload's cache (32 layers, 64 sequences x 8 KV heads, 2048
    store tokens + 64 residual) read by 32 query heads per sequence (r = 4),
    in the launch configuration the benchmark times; sampled (layer, sequence)
    pairs are compared with the oracle."""
    w = W.CONFIGS["batched_decode"]
    layers, batch, h_kv, r = w.layers, w.batch, w.kv_heads, 4
    bh = batch * h_kv
    r_cap, cap = 2 * w.residual, w.store_prefill + w.new_per_step
    cache = K.KiviCache(layers, bh, D, r_cap=r_cap, cap=cap, group=w.group, bits=w.bits,
                        residual=w.residual)
    fill_decode_store(w, cache, r_cap)
    q16 = queries(layers, batch, h_kv * r, 99)
    q = torch.from_numpy(q16.view(np.int16)).view(torch.float16).cuda()
    sc = 1.0 / math.sqrt(D)
    out = cache.decode_attention(q, batch, sm_scale=sc)
    torch.cuda.synchronize()
    assert K.kivi_device_fault() == 0
    got = out.cpu().numpy()
    n = w.store_prefill
    rng = np.random.default_rng(3)
    for l in rng.choice(layers, 3, replace=False):
        l = int(l)
        for b in rng.choice(batch, 3, replace=False):
            b = int(b)
            sl = dict(bh0=b * h_kv, bh=h_kv)
            kc, ks, kz = O.quantize_keys(W.generate(w, l, "k", n_tok=n, **sl), w.group, w.bits)
            vc, vs, vz = O.quantize_values(W.generate(w, l, "v", n_tok=n, **sl), w.group, w.bits)
            k = np.concatenate([O.dequantize_keys(kc, ks, kz, n, w.group, w.bits),
                                W.generate(w, l, "k", tok0=n, n_tok=r_cap, **sl)], axis=1)
            v = np.concatenate([O.dequantize_values(vc, vs, vz, w.group, w.bits),
                                W.generate(w, l, "v", tok0=n, n_tok=r_cap, **sl)], axis=1)
            ref = O.decode_attention(q16[l, b:b + 1].view(np.uint16), k, v, sc)[0]
            kf = k.view(np.float16).astype(np.float64)
            vf = v.view(np.float16).astype(np.float64)
            for h in range(h_kv * r):
                j = h // r
                qf = q16[l, b, h].astype(np.float64)
                s = sc * (kf[j] @ qf)
                p = np.exp(s - s.max())
                p /= p.sum()
                A = sc * np.max(np.abs(kf[j]) @ np.abs(qf))
                tol = (2.0 ** -16) * (1.0 + A) * (p @ np.abs(vf[j])) + 1e-30
                assert np.all(np.abs(got[l, b, h] - ref[h]) <= tol), (l, b, h)
