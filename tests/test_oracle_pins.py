"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Every function of ``oracle/`` is checked here against at least one of:
  * values printed on the pages (the flush sizes of the "Generation 1" table),
  * hand-worked examples built as the pages describe (inputs that land on .5,
    degenerate groups), stored under ``tests/golden/`` with their citations,
  * closed forms and special cases (integer inputs spanning exactly 2^b - 1,
    constant groups, the reconstruction error bound),
  * brute force in exact rational arithmetic on small inputs,
  * library routines for the binary16 conversions (numpy's float16),
  * a statistical figure the pages print (2-bit reconstruction cosine ~0.93),
  * an independent numpy re-derivation of the whole tensor path.
The sources are the VeloxQuant-MLX blog post "How I fused KIVI's KV-cache
quantization into two bit-exact Metal kernels ..." (the fused-kernel post),
the release post "VeloxQuant-MLX 0.8.0 adds KIVI" and the project README's
KIVI section.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _f16(values) -> np.ndarray:
    """binary16 bit patterns of decimal values that are exact in binary16."""
    a = np.array(values, dtype=np.float64)
    h = a.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), a) or np.all(np.isnan(a) == np.isnan(h))
    return h.view(np.uint16)


def unpack(words: np.ndarray, bits: int, axis: int) -> np.ndarray:
    """Codes from uint32 words, LSB first along ``axis`` (written from the
    packing definition, independent of the oracle)."""
    w = 32 // bits
    shifts = (np.arange(w, dtype=np.uint32) * bits)
    mask = np.uint32((1 << bits) - 1)
    q = (words[..., None] >> shifts) & mask          # [..., w] (axis expanded last)
    q = np.moveaxis(q, -1, axis + 1)                   # place the w codes after axis
    shape = list(words.shape)
    shape[axis] *= w
    return q.reshape(shape)


# ---------------------------------------------------------------------------
# binary16 conversions against numpy's float16
# ---------------------------------------------------------------------------

def test_half_to_float_all_65536_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = O.half_to_float(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_round_trip_ties_and_random():
    rng = np.random.default_rng(1)
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = h.view(np.float16).astype(np.float32)
    finite = np.isfinite(f)
    # every finite half survives a round trip, including -0 and subnormals
    assert np.array_equal(O.float_to_half(f[finite]), h[finite])
    # midpoints between neighbouring positive halves: exact in binary32,
    # ties go to the even neighbour; one binary32 ulp either side decides
    pos = h[(h >= 0) & (h < 0x7BFF)]
    lo = pos.view(np.float16).astype(np.float64)
    hi = (pos + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    cases = np.concatenate([mid, np.nextafter(mid, np.float32(0)),
                            np.nextafter(mid, np.float32(np.inf))])
    cases = np.concatenate([cases, -cases])
    # random magnitudes over every binade, the overflow edge and the underflow edge
    rnd = (rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 18, 200000))).astype(np.float32)
    edges = np.array([65504, 65519.996, 65520, 65536, 1e30, 2.0 ** -24, 2.0 ** -25,
                      2.0 ** -25 * 1.0000001, 2.0 ** -26, 1e-30, 0.0], np.float32)
    cases = np.concatenate([cases, rnd, edges, -edges]).astype(np.float32)
    got = O.float_to_half(cases)
    with np.errstate(over="ignore"):
        ref = cases.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# hand-worked groups (golden fixtures)
# ---------------------------------------------------------------------------

def _parse_ties():
    for line in _rows("rounding_ties.txt"):
        bits, vals, sz, codes, rec = [p.strip() for p in line.split("|")]
        yield (int(bits), [float(v) for v in vals.split()],
               [float(v) for v in sz.split()],
               [int(c.rstrip("*")) for c in codes.split()],
               [float(v) for v in rec.split()])


@pytest.mark.parametrize("row", list(_parse_ties()), ids=lambda r: f"b{r[0]}-{r[1][:3]}")
def test_rounding_ties_worked_examples(row):
    bits, vals, (scale_e, zero_e), codes_e, recon_e = row
    x = O.half_to_float(_f16(vals))
    scale, zero = O.group_params(x, bits)
    assert scale == np.float32(scale_e) and zero == np.float32(zero_e)
    codes = [O.code(v, scale, zero, bits) for v in x]
    assert codes == codes_e
    recon = [O.recon(q, scale, zero) for q in codes]
    assert recon == list(_f16(recon_e))


@pytest.mark.parametrize("row", list(_parse_ties()), ids=lambda r: f"b{r[0]}-{r[1][:3]}")
@pytest.mark.parametrize("group", [16, 32, 64])
def test_rounding_ties_through_tensor_paths(row, group):
    """The same worked examples, placed in a key group (token axis) and in a
    value group (channel axis) and padded by repeating their last value
    (which leaves min and max unchanged), come out of the full-tensor calls
    with the hand-worked codes at the right packed positions."""
    bits, vals, _, codes_e, recon_e = row
    n = len(vals)
    padded = vals + [vals[-1]] * (group - n)
    codes_full = codes_e + [codes_e[-1]] * (group - n)
    recon_full = recon_e + [recon_e[-1]] * (group - n)
    h = _f16(padded)
    # keys: one bh, `group` tokens, 8 identical channels
    xk = np.repeat(h[:, None], 8, axis=1)[None]
    c, s, z = O.quantize_keys(xk, group, bits)
    q = unpack(c, bits, axis=1)[0]
    assert np.array_equal(q, np.repeat(np.array(codes_full)[:, None], 8, axis=1))
    y = O.dequantize_keys(c, s, z, group, group, bits)
    assert np.array_equal(y[0, :, 0], _f16(recon_full))
    # values: one bh, 3 tokens, d = group channels
    xv = np.repeat(h[None, :], 3, axis=0)[None]
    c, s, z = O.quantize_values(xv, group, bits)
    q = unpack(c, bits, axis=2)[0]
    assert np.array_equal(q, np.repeat(np.array(codes_full)[None], 3, axis=0))
    y = O.dequantize_values(c, s, z, group, bits)
    assert np.array_equal(y[0, 1], _f16(recon_full))


def test_degenerate_groups():
    for line in _rows("degenerate_groups.txt"):
        bits, vals, sz, codes, rec = [p.strip() for p in line.split("|")]
        bits = int(bits)
        x = O.half_to_float(_f16([float(v) for v in vals.split()]))
        scale, zero = O.group_params(x, bits)
        sb, zb = [int(v, 16) for v in sz.split()]
        assert np.float32(scale).view(np.uint32) == sb
        assert np.float32(zero).view(np.uint32) == zb
        q = [O.code(v, scale, zero, bits) for v in x]
        assert q == [int(c) for c in codes.split()]
        assert [O.recon(c, scale, zero) for c in q] == [int(v, 16) for v in rec.split()]


def test_flush_sizes_match_generation1_table():
    for line in _rows("flush_sizes.txt"):
        prompt, residual, group, flushed = map(int, line.split())
        assert O.flush_size(prompt, residual, group) == flushed
        # the same through a real flush of a residual ring holding the prompt
        bh, d = 1, 32
        r_cap = -(-prompt // group) * group
        k = np.zeros((bh, r_cap, d), np.uint16)
        st = O.Store(bh, d, r_cap, group, 2)
        n, s_q, head, n_res = O.flush(k, k, st, residual, 0, 0, prompt)
        assert (n, s_q, head, n_res) == (flushed, flushed, flushed % r_cap, prompt - flushed)
        assert residual <= n_res < residual + group


def test_flush_size_rule_small_cases():
    # nothing moves until a whole group has aged past the window
    assert O.flush_size(0, 32, 32) == 0
    assert O.flush_size(63, 32, 32) == 0
    assert O.flush_size(64, 32, 32) == 32
    assert O.flush_size(95, 32, 32) == 32
    assert O.flush_size(96, 32, 32) == 64
    assert O.flush_size(127, 64, 64) == 0
    assert O.flush_size(128, 64, 64) == 64
    assert O.flush_size(40, 0, 32) == 32


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------

def test_8bit_integer_inputs_spanning_255_reconstruct_exactly():
    """With 2^b - 1 = 255 and integer inputs spanning exactly 255, scale is 1,
    every (x - zero) / scale is an integer and the reconstruction is exact."""
    rng = np.random.default_rng(7)
    bh, s, d, g = 2, 64, 64, 32
    base = rng.integers(-300, 300, size=(bh, s // g, 1, d))
    x = base + rng.integers(0, 256, size=(bh, s // g, g, d))
    x[:, :, 0, :] = base[:, :, 0, :]            # min of every key group
    x[:, :, 1, :] = base[:, :, 0, :] + 255      # max of every key group
    xk = _f16(x.reshape(bh, s, d))
    c, sc, ze = O.quantize_keys(xk, g, 8)
    assert np.all(sc == 1.0)
    assert np.array_equal(O.dequantize_keys(c, sc, ze, s, g, 8), xk)
    # values: every channel group of a token spans exactly 255
    xv = x.reshape(bh, s, d).copy()
    for gi in range(d // g):
        blk = xv[:, :, gi * g:(gi + 1) * g]
        blk[...] = blk[:, :, :1] + (blk - blk[:, :, :1]) % 256
        blk[:, :, 1] = blk[:, :, 0] + 255
        blk[:, :, 2:] = np.minimum(blk[:, :, 2:], blk[:, :, :1] + 255)
        blk[...] = np.maximum(blk, blk[:, :, :1])
    xv16 = _f16(xv)
    c, sc, ze = O.quantize_values(xv16, g, 8)
    assert np.all(sc == 1.0)
    assert np.array_equal(O.dequantize_values(c, sc, ze, g, 8), xv16)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_constant_groups_reconstruct_exactly(bits):
    rng = np.random.default_rng(bits)
    vals = rng.standard_normal((2, 1, 96)) * 5
    x = _f16(np.repeat(vals.astype(np.float16).astype(np.float64), 64, axis=1))  # [2, 64, 96]
    c, s, z = O.quantize_keys(x, 32, bits)
    assert np.all(s == 0) and np.all(c == 0)
    assert np.array_equal(O.dequantize_keys(c, s, z, 64, 32, bits), x)
    xt = np.ascontiguousarray(np.swapaxes(x, 1, 2))[:, :, :64]    # constant along channels
    xt = np.ascontiguousarray(np.repeat(xt[:, :, :1], 64, axis=2))
    c, s, z = O.quantize_values(xt, 32, bits)
    assert np.all(s == 0) and np.all(c == 0)
    assert np.array_equal(O.dequantize_values(c, s, z, 32, bits), xt)


# ---------------------------------------------------------------------------
# invariants and brute force on seeded workloads
# ---------------------------------------------------------------------------

SHAPES = [  # (bh, s, d, group, bits)
    (3, 96, 128, 32, 2), (2, 100, 64, 32, 4), (2, 77, 128, 64, 8),
    (1, 130, 128, 128, 2), (2, 64, 256, 64, 4), (1, 5, 32, 32, 8),
    (2, 50, 64, 16, 2), (1, 40, 96, 16, 4), (2, 37, 32, 16, 8),
]


def _input(bh, s, d, seed, kind):
    w = W.custom(seed=seed, batch=1, kv_heads=bh, seq=s, head_dim=d)
    return W.generate(w, 0, kind)


def _exact_nearest(r: Fraction, qmax: int) -> int:
    k = min(range(qmax + 1), key=lambda j: (abs(r - j), j % 2))
    return k


@pytest.mark.parametrize("shape", SHAPES, ids=str)
def test_key_invariants(shape):
    bh, s, d, g, bits = shape
    Q = (1 << bits) - 1
    x = _input(bh, s, d, 11 + s, "k")
    xf = x.view(np.float16).astype(np.float64)
    c, sc, ze = O.quantize_keys(x, g, bits)
    ng = -(-s // g)
    assert c.shape == (bh, ng * g // (32 // bits), d) and sc.shape == (bh, ng, d)
    q = unpack(c, bits, axis=1)                              # [bh, ng*g, d]
    # edge-replicated view of the input (padding semantics)
    idx = np.minimum(np.arange(ng * g), s - 1)
    xp = xf[:, idx, :].reshape(bh, ng, g, d)
    qg = q.reshape(bh, ng, g, d)
    mn, mx = xp.min(axis=2), xp.max(axis=2)
    # zero is the group minimum along the token axis, per channel
    assert np.array_equal(ze.astype(np.float64), mn + 0.0)
    pos = sc > 0
    # the minimum maps to code 0 and the maximum to 2^b - 1
    assert np.all(qg[xp == mn[:, :, None, :]] == 0)
    at_max = (xp == mx[:, :, None, :]) & pos[:, :, None, :]
    assert np.all(qg[at_max] == Q)
    assert np.all(q <= Q)
    # codes of padded slots repeat the code of the last token
    if s % g:
        assert np.all(q[:, s:, :] == q[:, s - 1:s, :])
    # reconstruction within half a step plus binary32 and binary16 rounding
    y = O.dequantize_keys(c, sc, ze, s, g, bits).view(np.float16).astype(np.float64)
    step = np.repeat(sc.astype(np.float64), g, axis=1)[:, :s, :]
    zz = np.repeat(ze.astype(np.float64), g, axis=1)[:, :s, :]
    ulp16 = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64)
    bound = step / 2 * (1 + 2.0 ** -20) + 2.0 ** -22 * (np.abs(zz) + np.abs(xf) + np.abs(y)) + ulp16 / 2
    assert np.all(np.abs(xf - y) <= bound)
    # each group agrees with the single-group oracle call (layout check)
    rng = np.random.default_rng(s)
    for _ in range(8):
        b, gi, ch = rng.integers(bh), rng.integers(ng), rng.integers(d)
        words, s1, z1 = O.key_group(x[b], gi, ch, g, bits)
        per = g // (32 // bits)
        assert np.array_equal(words, c[b, gi * per:(gi + 1) * per, ch])
        assert s1 == sc[b, gi, ch] and z1 == ze[b, gi, ch]


@pytest.mark.parametrize("shape", SHAPES, ids=str)
def test_value_invariants(shape):
    bh, s, d, g, bits = shape
    Q = (1 << bits) - 1
    x = _input(bh, s, d, 29 + s, "v")
    xf = x.view(np.float16).astype(np.float64)
    c, sc, ze = O.quantize_values(x, g, bits)
    assert c.shape == (bh, s, d // (32 // bits)) and sc.shape == (bh, s, d // g)
    q = unpack(c, bits, axis=2)
    xg = xf.reshape(bh, s, d // g, g)
    qg = q.reshape(bh, s, d // g, g)
    mn, mx = xg.min(axis=3), xg.max(axis=3)
    # zero is the group minimum along the channel axis, per token
    assert np.array_equal(ze.astype(np.float64), mn + 0.0)
    assert np.all(qg[xg == mn[..., None]] == 0)
    assert np.all(qg[(xg == mx[..., None]) & (sc[..., None] > 0)] == Q)
    y = O.dequantize_values(c, sc, ze, g, bits).view(np.float16).astype(np.float64)
    step = np.repeat(sc.astype(np.float64), g, axis=2)
    zz = np.repeat(ze.astype(np.float64), g, axis=2)
    ulp16 = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64)
    bound = step / 2 * (1 + 2.0 ** -20) + 2.0 ** -22 * (np.abs(zz) + np.abs(xf) + np.abs(y)) + ulp16 / 2
    assert np.all(np.abs(xf - y) <= bound)
    rng = np.random.default_rng(s)
    for _ in range(8):
        b, t = rng.integers(bh), rng.integers(s)
        words, s1, z1 = O.value_row(x[b, t], g, bits)
        assert np.array_equal(words, c[b, t]) and np.array_equal(s1, sc[b, t])
        assert np.array_equal(z1, ze[b, t])


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_brute_force_exact_rationals(bits):
    """Every code is the nearest grid index to (x - zero) / scale, found by
    enumerating all 2^b candidates in exact rational arithmetic; ties go to
    the even index.  Only where the exact ratio lies within binary32 rounding
    of a half-integer may the rounded computation pick the neighbour, and
    then it must agree with the enumeration over the binary32 quotient.
    The sample is chosen to include such near-ties."""
    Q = (1 << bits) - 1
    x = _input(2, 40, 64, 300 + bits, "k")
    c, sc, ze = O.quantize_keys(x, 32, bits)
    q = unpack(c, bits, axis=1)
    xf = x.view(np.float16).astype(np.float32)
    for b in range(2):
        for t in range(40):
            for ch in range(0, 64, 3):
                gi = t // 32
                s_, z_ = sc[b, gi, ch], ze[b, gi, ch]
                got = int(q[b, t, ch])
                if s_ == 0:
                    assert got == 0
                    continue
                r = (Fraction(float(xf[b, t, ch])) - Fraction(float(z_))) / Fraction(float(s_))
                k = _exact_nearest(r, Q)
                frac_dist = abs(abs(r - int(r)) - Fraction(1, 2))
                # binary32 rounding of (x - zero) and of the quotient moves the
                # ratio by at most 2 * 2^-24 relative; stay well clear of that
                if frac_dist > abs(r) * Fraction(1, 1 << 21) + Fraction(1, 1 << 40):
                    assert got == k, (b, t, ch, float(r))
                else:
                    u = np.float32(np.float32(xf[b, t, ch] - z_) / s_)
                    assert got == _exact_nearest(Fraction(float(u)), Q)


def test_permuting_tokens_in_a_group_permutes_codes_only():
    x = _input(2, 64, 64, 5, "k")
    c, s, z = O.quantize_keys(x, 32, 2)
    rng = np.random.default_rng(3)
    perm = np.concatenate([rng.permutation(32), 32 + rng.permutation(32)])
    c2, s2, z2 = O.quantize_keys(np.ascontiguousarray(x[:, perm]), 32, 2)
    assert np.array_equal(s, s2) and np.array_equal(z, z2)
    assert np.array_equal(unpack(c, 2, 1)[:, perm], unpack(c2, 2, 1))


def test_determinism():
    x = _input(2, 96, 128, 8, "v")
    a = O.quantize_values(x, 32, 4)
    b = O.quantize_values(x.copy(), 32, 4)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))


def test_product_is_rounded_before_the_add():
    """The reconstruction rounds q*scale to binary32 before adding zero (the
    fused-kernel post, "1. FMA contraction": separate multiply and add, two
    roundings).  Find inputs where a fused multiply-add would give a
    different binary16 result, using exact rationals for the fused value,
    and check the oracle returns the two-rounding value."""
    rng = np.random.default_rng(123)
    n = 400000
    q = rng.integers(1, 4, n).astype(np.float32)
    s = (rng.uniform(0.05, 3, n)).astype(np.float32)
    z = (-rng.uniform(0, 4, n)).astype(np.float32)
    two = ((q * s) + z).astype(np.float32)
    fused = (q.astype(np.float64) * s.astype(np.float64) + z.astype(np.float64))
    # the double sum is exact when the two addends are within 2^27 of each other
    fused32 = fused.astype(np.float32)
    cand = np.nonzero(two.astype(np.float16) != fused32.astype(np.float16))[0]
    checked = 0
    for i in cand[:50]:
        exact = Fraction(float(q[i])) * Fraction(float(s[i])) + Fraction(float(z[i]))
        if Fraction(float(fused[i])) != exact:
            continue
        checked += 1
        got = O.recon(int(q[i]), s[i], z[i])
        assert got == two[i].astype(np.float16).view(np.uint16)
        assert got != fused32[i].astype(np.float16).view(np.uint16)
    assert checked > 0


def test_two_bit_reconstruction_cosine_on_unit_norm_gaussian_keys():
    """Release post "Honest limitations" and the README's KIVI section: at 2
    bits, the reconstruction cosine of synthetic unit-norm Gaussian keys sits
    around 0.93 (defaults G=32, keys per channel)."""
    w = W.custom(seed=77, batch=1, kv_heads=16, seq=1024, head_dim=128,
                 keys=W.Dist(W.NORMAL, 1.0))
    k = W.generate(w, 0, "k").view(np.float16).astype(np.float64)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    x = k.astype(np.float16).view(np.uint16)
    c, s, z = O.quantize_keys(x, 32, 2)
    y = O.dequantize_keys(c, s, z, 1024, 32, 2).view(np.float16).astype(np.float64)
    xf = x.view(np.float16).astype(np.float64)
    cos = np.sum(xf * y, -1) / np.linalg.norm(xf, axis=-1) / np.linalg.norm(y, axis=-1)
    assert abs(cos.mean() - 0.93) < 0.01, cos.mean()


# ---------------------------------------------------------------------------
# independent numpy re-derivation
# ---------------------------------------------------------------------------

def _np_group_quant(xg: np.ndarray, axis: int, bits: int):
    """numpy binary32 version of the quantizer: one IEEE operation per ufunc."""
    Q = np.float32((1 << bits) - 1)
    mn = xg.min(axis=axis, keepdims=True) + np.float32(0)
    mx = xg.max(axis=axis, keepdims=True) + np.float32(0)
    scale = (mx - mn) / Q
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (xg - mn) / scale
    q = np.where(scale == 0, np.float32(0), np.clip(np.rint(u), 0, Q)).astype(np.uint32)
    return q, scale, mn


def _np_pack(q: np.ndarray, bits: int, axis: int) -> np.ndarray:
    w = 32 // bits
    q = np.moveaxis(q, axis, -1)
    q = q.reshape(q.shape[:-1] + (q.shape[-1] // w, w)).astype(np.uint32)
    words = np.bitwise_or.reduce(q << (np.arange(w, dtype=np.uint32) * bits), axis=-1)
    return np.moveaxis(words, -1, axis)


REDERIVE = {"tiny_flush": W.CONFIGS["tiny_flush"],
            "g16_b4": W.custom(seed=12, kv_heads=3, seq=80, head_dim=64, bits=4, group=16),
            "g16_b2": W.custom(seed=13, kv_heads=2, seq=48, head_dim=128, bits=2, group=16)}


@pytest.mark.parametrize("name", sorted(REDERIVE))
def test_numpy_rederivation_matches_oracle_bit_for_bit(name):
    w = REDERIVE[name]
    g, bits = w.group, w.bits
    for kind in ("k", "v"):
        x = W.generate(w, 0, kind)
        bh, s, d = x.shape
        xf = x.view(np.float16).astype(np.float32)
        if kind == "k":
            q, sc, ze = _np_group_quant(xf.reshape(bh, s // g, g, d), 2, bits)
            words = _np_pack(q.reshape(bh, s, d), bits, 1)
            sc, ze = sc[:, :, 0, :], ze[:, :, 0, :]
            oc, osc, oze = O.quantize_keys(x, g, bits)
            prod = q.astype(np.float32) * sc[:, :, None, :]
            y = (prod + ze[:, :, None, :]).astype(np.float16).view(np.uint16).reshape(bh, s, d)
            oy = O.dequantize_keys(oc, osc, oze, s, g, bits)
        else:
            q, sc, ze = _np_group_quant(xf.reshape(bh, s, d // g, g), 3, bits)
            words = _np_pack(q.reshape(bh, s, d), bits, 2)
            sc, ze = sc[..., 0], ze[..., 0]
            oc, osc, oze = O.quantize_values(x, g, bits)
            prod = q.astype(np.float32) * sc[..., None]
            y = (prod + ze[..., None]).astype(np.float16).view(np.uint16).reshape(bh, s, d)
            oy = O.dequantize_values(oc, osc, oze, g, bits)
        assert np.array_equal(words, oc)
        assert np.array_equal(sc.view(np.uint32), osc.view(np.uint32))
        assert np.array_equal(ze.view(np.uint32), oze.view(np.uint32))
        assert np.array_equal(y, oy)


# ---------------------------------------------------------------------------
# flush bookkeeping
# ---------------------------------------------------------------------------

def test_flush_sequence_with_ring_wrap_equals_full_quantization():
    """Prefill then decode steps through a small ring: the store ends up
    holding exactly the full-tensor quantization of every flushed token, and
    the residual keeps the newest tokens in order."""
    G, R, bits, bh, d = 32, 32, 2, 3, 64
    total = 64 + 7 * 16
    w = W.custom(seed=9, batch=1, kv_heads=bh, seq=total, head_dim=d)
    K = W.generate(w, 0, "k")
    V = W.generate(w, 0, "v")
    r_cap, cap = 96, 256
    k_res = np.zeros((bh, r_cap, d), np.uint16)
    v_res = np.zeros((bh, r_cap, d), np.uint16)
    st = O.Store(bh, d, cap, G, bits)
    s_q, head, n_res, pos = 0, 0, 0, 0

    def append(n):
        nonlocal n_res, pos
        for i in range(n):
            row = (head + n_res) % r_cap
            k_res[:, row] = K[:, pos]
            v_res[:, row] = V[:, pos]
            n_res += 1
            pos += 1

    append(64)
    flushed = []
    n, s_q, head, n_res = O.flush(k_res, v_res, st, R, s_q, head, n_res)
    flushed.append(n)
    while pos < total:
        append(16)
        n, s_q, head, n_res = O.flush(k_res, v_res, st, R, s_q, head, n_res)
        flushed.append(n)
    assert flushed == [32, 0, 32, 0, 32, 0, 32, 0]
    assert s_q == 128 and n_res == total - 128 and R <= n_res < R + G
    ck, sk, zk = O.quantize_keys(np.ascontiguousarray(K[:, :s_q]), G, bits)
    cv, sv, zv = O.quantize_values(np.ascontiguousarray(V[:, :s_q]), G, bits)
    w_ = 32 // bits
    assert np.array_equal(st.k_codes[:, :s_q // w_], ck)
    assert np.array_equal(st.k_scale[:, :s_q // G], sk) and np.array_equal(st.k_zero[:, :s_q // G], zk)
    assert np.array_equal(st.v_codes[:, :s_q], cv)
    assert np.array_equal(st.v_scale[:, :s_q], sv) and np.array_equal(st.v_zero[:, :s_q], zv)
    # the residual holds the newest tokens, oldest first, starting at head
    rows = (head + np.arange(n_res)) % r_cap
    assert np.array_equal(k_res[:, rows], K[:, s_q:total])


def test_flush_sequence_g16_odd_ring_equals_full_quantization():
    """The same at G = 16 with a ring of 80 rows (not a multiple of 32), so
    groups start at every multiple of 16 and the ring wraps mid-way."""
    G, R, bits, bh, d = 16, 16, 4, 2, 32
    total = 64 + 9 * 16
    w = W.custom(seed=19, batch=1, kv_heads=bh, seq=total, head_dim=d)
    K = W.generate(w, 0, "k")
    V = W.generate(w, 0, "v")
    r_cap, cap = 80, 256
    k_res = np.zeros((bh, r_cap, d), np.uint16)
    v_res = np.zeros((bh, r_cap, d), np.uint16)
    st = O.Store(bh, d, cap, G, bits)
    s_q, head, n_res, pos = 0, 0, 0, 0
    flushed = []
    for n_new in [64] + [16] * 9:
        for _ in range(n_new):
            row = (head + n_res) % r_cap
            k_res[:, row] = K[:, pos]
            v_res[:, row] = V[:, pos]
            n_res += 1
            pos += 1
        n, s_q, head, n_res = O.flush(k_res, v_res, st, R, s_q, head, n_res)
        flushed.append(n)
    assert flushed == [48] + [16] * 9
    assert s_q == total - 16 and n_res == 16 and head == s_q % r_cap
    ck, sk, zk = O.quantize_keys(np.ascontiguousarray(K[:, :s_q]), G, bits)
    cv, sv, zv = O.quantize_values(np.ascontiguousarray(V[:, :s_q]), G, bits)
    w_ = 32 // bits
    assert np.array_equal(st.k_codes[:, :s_q // w_], ck)
    assert np.array_equal(st.k_scale[:, :s_q // G], sk) and np.array_equal(st.k_zero[:, :s_q // G], zk)
    assert np.array_equal(st.v_codes[:, :s_q], cv)
    assert np.array_equal(st.v_scale[:, :s_q], sv) and np.array_equal(st.v_zero[:, :s_q], zv)


def test_append_places_tokens_in_ring_order():
    """The oracle's append against a token-by-token placement written here
    (the sequence's token j at ring row (head + its residual index) mod
    r_cap), over chunk sizes that wrap the ring mid-chunk, interleaved with
    flushes; the flushed store ends up holding exactly the full quantization
    of every flushed token, and the residual the newest tokens in order."""
    G, R, bits, bh, d = 32, 32, 4, 2, 64
    chunks = [64, 16, 16, 5, 27, 16, 30, 2, 40, 1, 31, 33]
    total = sum(chunks)
    w = W.custom(seed=29, batch=1, kv_heads=bh, seq=total, head_dim=d)
    K = W.generate(w, 0, "k")
    V = W.generate(w, 0, "v")
    r_cap, cap = 96, 512
    k_res = np.zeros((bh, r_cap, d), np.uint16)
    v_res = np.zeros((bh, r_cap, d), np.uint16)
    k_ref, v_ref = k_res.copy(), v_res.copy()
    st = O.Store(bh, d, cap, G, bits)
    s_q, head, n_res, pos = 0, 0, 0, 0
    wrapped = False
    for n_new in chunks:
        assert n_res + n_new <= r_cap
        for j in range(n_new):                      # the placement by its definition
            row = (head + n_res + j) % r_cap
            wrapped |= row < (head + n_res) % r_cap
            k_ref[:, row] = K[:, pos + j]
            v_ref[:, row] = V[:, pos + j]
        n_res2 = O.append(k_res, v_res, head, n_res, K[:, pos:pos + n_new], V[:, pos:pos + n_new])
        assert n_res2 == n_res + n_new
        assert np.array_equal(k_res, k_ref) and np.array_equal(v_res, v_ref)
        n_res, pos = n_res2, pos + n_new
        _, s_q, head, n_res = O.flush(k_res, v_res, st, R, s_q, head, n_res)
    assert wrapped and s_q >= 192
    ck, sk, zk = O.quantize_keys(np.ascontiguousarray(K[:, :s_q]), G, bits)
    cv, sv, zv = O.quantize_values(np.ascontiguousarray(V[:, :s_q]), G, bits)
    w_ = 32 // bits
    assert np.array_equal(st.k_codes[:, :s_q // w_], ck)
    assert np.array_equal(st.k_scale[:, :s_q // G], sk) and np.array_equal(st.k_zero[:, :s_q // G], zk)
    assert np.array_equal(st.v_codes[:, :s_q], cv)
    assert np.array_equal(st.v_scale[:, :s_q], sv) and np.array_equal(st.v_zero[:, :s_q], zv)
    rows = (head + np.arange(n_res)) % r_cap
    assert np.array_equal(k_res[:, rows], K[:, s_q:total])
    assert np.array_equal(v_res[:, rows], V[:, s_q:total])


def test_append_rejects_ring_overflow():
    bh, d, r_cap = 1, 32, 64
    k = np.zeros((bh, r_cap, d), np.uint16)
    v = np.zeros((bh, r_cap, d), np.uint16)
    new = np.ones((bh, 40, d), np.uint16)
    assert O.append(k, v, 0, 20, new, new) == 60
    with pytest.raises(ValueError):
        O.append(k, v, 0, 30, new, new)           # 70 tokens in a 64-row ring
    with pytest.raises(ValueError):
        O.append(k, v, 64, 0, new, new)           # head outside the ring


def test_flush_rejects_overflowing_store_and_bad_state():
    bh, d = 1, 32
    k = np.zeros((bh, 128, d), np.uint16)
    st = O.Store(bh, d, 64, 32, 2)
    with pytest.raises(ValueError):
        O.flush(k, k, st, 32, 0, 0, 128)          # 96 tokens into a 64-token store
    with pytest.raises(ValueError):
        O.flush(k, k, st, 32, 16, 0, 64)          # store offset not a multiple of G
    with pytest.raises(ValueError):
        O.flush(k, k, st, 32, 0, 0, 129)          # more residual than the ring holds
