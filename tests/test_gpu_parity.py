"""Bit-exact parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every output element: packed codes, binary32 scale and
zero (as bit patterns) and binary16 reconstructions.  They span several
tiles, ragged tails, every (bits, group) pair, odd head dims and the
degenerate inputs the method has (constant groups, signed zeros, exact .5
ties, subnormals, extremes, groups far from zero).  Full-size workloads run
in the launch configuration the benchmark times and are checked on sampled
groups that the oracle computes one by one, plus one complete layer (the
last) of each prefill and one complete bh slice (the last) of every store
sweep cell, for all four kernels and the fused forms.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import (assert_same, bits32, hard_block, host_f32_bits, host_u16, host_u32,
                      sample_keys, sample_values, to_dev)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_cache_quantization_kivi_gb300 as K  # noqa: E402

COMBOS = [(b, g) for b in (2, 4, 8) for g in (16, 32, 64, 128)]


# ---------------------------------------------------------------------------
# full-tensor calls against the full oracle
# ---------------------------------------------------------------------------

def gpu_keys(x: np.ndarray, group: int, bits: int):
    xd = to_dev(x)
    c, s, z = K.kivi_quantize_keys(xd, group, bits)
    y = K.kivi_dequantize_keys(c, s, z, x.shape[1], group, bits)
    torch.cuda.synchronize()
    return host_u32(c), host_f32_bits(s), host_f32_bits(z), host_u16(y)


def gpu_values(x: np.ndarray, group: int, bits: int):
    xd = to_dev(x)
    c, s, z = K.kivi_quantize_values(xd, group, bits)
    y = K.kivi_dequantize_values(c, s, z, group, bits)
    torch.cuda.synchronize()
    return host_u32(c), host_f32_bits(s), host_f32_bits(z), host_u16(y)


def check_keys(x: np.ndarray, group: int, bits: int) -> None:
    c, s, z, y = gpu_keys(x, group, bits)
    oc, os_, oz = O.quantize_keys(x, group, bits)
    oy = O.dequantize_keys(oc, os_, oz, x.shape[1], group, bits)
    assert_same("key codes", c, oc)
    assert_same("key scale", s, bits32(os_))
    assert_same("key zero", z, bits32(oz))
    assert_same("key recon", y, oy)


def check_values(x: np.ndarray, group: int, bits: int) -> None:
    c, s, z, y = gpu_values(x, group, bits)
    oc, os_, oz = O.quantize_values(x, group, bits)
    oy = O.dequantize_values(oc, os_, oz, group, bits)
    assert_same("value codes", c, oc)
    assert_same("value scale", s, bits32(os_))
    assert_same("value zero", z, bits32(oz))
    assert_same("value recon", y, oy)


def _x(bh, s, d, seed, kind, keys=None):
    w = W.custom(seed=seed, batch=1, kv_heads=bh, seq=s, head_dim=d,
                 keys=keys or W.Dist(W.NORMAL, 1.0, n_outliers=min(4, d), outlier_mult=15.0))
    return W.generate(w, 0, kind)


@pytest.fixture(params=["register", "staged"])
def key_quantizer(request, monkeypatch):
    """Runs a test on both key quantizers, forced by KIVI_KEY_QUANTIZER
    (read by the library at each call): the register kernel and the staged
    one (which takes head_dim 128 at G >= 32 in plain mode; the register
    kernel keeps the rest).  Without the variable the library picks by G and
    width."""
    monkeypatch.setenv("KIVI_KEY_QUANTIZER", request.param)
    return request.param


@pytest.mark.parametrize("bits,group", COMBOS)
def test_keys_several_tiles_ragged_tail(bits, group, key_quantizer):
    check_keys(_x(3, 3 * group + 5, 128, 1000 + bits * group, "k"), group, bits)


@pytest.mark.parametrize("bits,group", COMBOS)
def test_values_several_rows(bits, group):
    check_values(_x(3, 77, 128, 2000 + bits * group, "v"), group, bits)


@pytest.mark.parametrize("shape", [
    (1, 1, 128, 32, 2), (2, 5, 64, 64, 4), (1, 200, 8, 32, 2), (2, 100, 40, 64, 8),
    (1, 129, 256, 128, 2), (4, 64, 256, 32, 4), (2, 300, 16, 128, 8), (5, 31, 128, 32, 2),
    (2, 37, 64, 16, 2), (1, 17, 8, 16, 8), (3, 100, 40, 16, 4), (1, 1, 256, 16, 2),
], ids=str)
def test_keys_odd_shapes(shape, key_quantizer):
    bh, s, d, g, b = shape
    check_keys(_x(bh, s, d, 3000 + s + d, "k"), g, b)


@pytest.mark.parametrize("shape", [
    (1, 1, 32, 32, 2), (2, 50, 96, 32, 4), (1, 33, 256, 128, 8), (2, 64, 192, 64, 2),
    (1, 40, 64, 64, 8), (7, 3, 128, 128, 4),
    (2, 19, 96, 16, 2), (1, 5, 256, 16, 8), (3, 33, 32, 16, 4),
], ids=str)
def test_values_odd_shapes(shape):
    bh, s, d, g, b = shape
    check_values(_x(bh, s, d, 4000 + s + d, "v"), g, b)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits,group", COMBOS)
def test_keys_degenerate_and_tie_groups(bits, group, d, key_quantizer):
    rng = np.random.default_rng(bits * 7 + group + d)
    bh = 2
    blocks = [hard_block(rng, group, d) for _ in range(bh * 3)]
    x = np.stack([np.concatenate(blocks[3 * b:3 * b + 3], axis=0) for b in range(bh)])
    check_keys(x.astype(np.float16).view(np.uint16), group, bits)


@pytest.mark.parametrize("bits,group", COMBOS)
def test_values_degenerate_and_tie_groups(bits, group):
    rng = np.random.default_rng(bits * 11 + group)
    bh, s, d = 2, 40, 2 * group
    x = np.stack([np.concatenate([hard_block(rng, group, s).T for _ in range(d // group)], axis=1)
                  for _ in range(bh)])
    check_values(x.astype(np.float16).view(np.uint16), group, bits)


def test_strided_inputs_and_outputs(key_quantizer):
    bh, s, d, g, b = 3, 96, 128, 32, 4
    x = _x(bh, s, d, 55, "k")
    big = torch.zeros((bh, s + 40, d), dtype=torch.float16, device="cuda")
    big[:, :s] = to_dev(x)
    xv = big[:, :s]                                     # bh stride (s + 40) * d
    ng = s // g
    codes = torch.zeros((bh, ng * g // (32 // b) + 4, d), dtype=torch.int32, device="cuda")
    scale = torch.zeros((bh, ng + 2, d), dtype=torch.float32, device="cuda")
    zero = torch.zeros((bh, ng + 2, d), dtype=torch.float32, device="cuda")
    K.kivi_quantize_keys(xv, g, b, codes[:, :ng * g // (32 // b)], scale[:, :ng], zero[:, :ng])
    y = torch.zeros((bh, s + 8, d), dtype=torch.float16, device="cuda")
    K.kivi_dequantize_keys(codes[:, :ng * g // (32 // b)], scale[:, :ng], zero[:, :ng], s, g, b,
                           y[:, :s])
    torch.cuda.synchronize()
    oc, os_, oz = O.quantize_keys(x, g, b)
    assert_same("codes", host_u32(codes[:, :ng * g // (32 // b)]), oc)
    assert not host_u32(codes[:, ng * g // (32 // b):]).any()      # padding untouched
    assert_same("scale", host_f32_bits(scale[:, :ng]), bits32(os_))
    assert_same("recon", host_u16(y[:, :s]), O.dequantize_keys(oc, os_, oz, s, g, b))
    assert not host_u16(y[:, s:]).any()


def test_empty_calls_are_noops():
    x = torch.zeros((0, 64, 128), dtype=torch.float16, device="cuda")
    c, s, z = K.kivi_quantize_keys(x, 32, 2)
    assert c.numel() == 0
    x = torch.zeros((2, 0, 128), dtype=torch.float16, device="cuda")
    K.kivi_quantize_values(x, 32, 2)
    torch.cuda.synchronize()


def test_determinism():
    x = _x(4, 257, 128, 77, "k")
    a = gpu_keys(x, 64, 4)
    b = gpu_keys(x, 64, 4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_tiny_flush_config_end_to_end(key_quantizer):
    """The tiny flush workload: 8 heads x 128 tokens, 2-bit, G=R=32; the flush
    moves 96 tokens and keeps 32 in fp16; keys and values also quantized as
    full tensors."""
    w = W.CONFIGS["tiny_flush"]
    k = W.generate(w, 0, "k")
    v = W.generate(w, 0, "v")
    check_keys(k, w.group, w.bits)
    check_values(v, w.group, w.bits)
    cache = K.KiviCache(1, w.bh, w.head_dim, r_cap=128, cap=128, group=w.group, bits=w.bits,
                        residual=w.residual)
    cache.append(0, to_dev(k), to_dev(v))
    cache.advance(128)
    assert cache.flush() == 96
    st = O.Store(w.bh, w.head_dim, 128, w.group, w.bits)
    n, s_q, head, n_res = O.flush(k, v, st, w.residual, 0, 0, 128)
    assert (n, s_q, head, n_res) == (96, cache.s_q, cache.res_head, cache.n_res)
    torch.cuda.synchronize()
    compare_store(cache, 0, st)
    ky, vy = cache.dequantize()
    torch.cuda.synchronize()
    assert_same("key recon", host_u16(ky[0]),
                O.dequantize_keys(st.k_codes[:, :96 // 16], st.k_scale[:, :3], st.k_zero[:, :3],
                                  96, w.group, w.bits))
    assert_same("value recon", host_u16(vy[0]),
                O.dequantize_values(st.v_codes[:, :96], st.v_scale[:, :96], st.v_zero[:, :96],
                                    w.group, w.bits))


def compare_store(cache, layer: int, st) -> None:
    assert_same("store key codes", host_u32(cache.k_codes[layer]), st.k_codes)
    assert_same("store key scale", host_f32_bits(cache.k_scale[layer]), bits32(st.k_scale))
    assert_same("store key zero", host_f32_bits(cache.k_zero[layer]), bits32(st.k_zero))
    assert_same("store value codes", host_u32(cache.v_codes[layer]), st.v_codes)
    assert_same("store value scale", host_f32_bits(cache.v_scale[layer]), bits32(st.v_scale))
    assert_same("store value zero", host_f32_bits(cache.v_zero[layer]), bits32(st.v_zero))


@pytest.mark.parametrize("bits,group,residual", [(4, 32, 32), (8, 64, 64), (2, 128, 32),
                                                  (2, 16, 16), (8, 16, 32)])
def test_multi_layer_flush_sequence_with_ring_wrap(bits, group, residual, key_quantizer):
    layers, bh, d = 3, 4, 128
    r_cap = 3 * group + (residual // group + 1) * group
    cap = 16 * group
    total = 14 * group
    w = W.custom(seed=60 + bits, batch=1, kv_heads=bh, seq=total, head_dim=d)
    K_all = [W.generate(w, l, "k") for l in range(layers)]
    V_all = [W.generate(w, l, "v") for l in range(layers)]
    cache = K.KiviCache(layers, bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                        residual=residual)
    ring_k = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    ring_v = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    stores = [O.Store(bh, d, cap, group, bits) for _ in range(layers)]
    s_q = head = n_res = pos = 0
    rng = np.random.default_rng(bits)
    flushed = 0
    while pos < total:
        n_new = int(min(total - pos, rng.integers(1, 2 * group)))
        n_new = min(n_new, r_cap - n_res)
        rows = (head + n_res + np.arange(n_new)) % r_cap
        for l in range(layers):
            ring_k[l][:, rows] = K_all[l][:, pos:pos + n_new]
            ring_v[l][:, rows] = V_all[l][:, pos:pos + n_new]
            cache.append(l, to_dev(K_all[l][:, pos:pos + n_new]),
                         to_dev(V_all[l][:, pos:pos + n_new]))
        cache.advance(n_new)
        n_res += n_new
        pos += n_new
        n_gpu = cache.flush()
        for l in range(layers):
            n, s_q2, head2, n_res2 = O.flush(ring_k[l], ring_v[l], stores[l], residual,
                                              s_q, head, n_res)
        s_q, head, n_res = s_q2, head2, n_res2
        assert n_gpu == n and (cache.s_q, cache.res_head, cache.n_res) == (s_q, head, n_res)
        flushed += n
    assert flushed >= 8 * group
    torch.cuda.synchronize()
    for l in range(layers):
        compare_store(cache, l, stores[l])


# ---------------------------------------------------------------------------
# full-size workloads, sampled against per-group oracle calls
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama3_2_3b_prefill", "qwen2_5_7b_long"])
def test_prefill_flush_full_size_sampled(name, key_quantizer):
    """All layers' residual windows hold the whole prompt; one flush (one
    launch per tensor kind over every layer) moves all but the newest
    tokens; the store is then dequantized in one launch per kind."""
    w = W.CONFIGS[name]
    cache = K.KiviCache(w.layers, w.bh, w.head_dim, r_cap=w.seq, cap=w.seq, group=w.group,
                        bits=w.bits, residual=w.residual)
    hosts = []
    for l in range(w.layers):
        k = W.generate(w, l, "k")
        v = W.generate(w, l, "v")
        cache.k_res[l].copy_(to_dev(k))
        cache.v_res[l].copy_(to_dev(v))
        hosts.append((k, v))
    cache.advance(w.seq)
    n = cache.flush()
    assert n == O.flush_size(w.seq, w.residual, w.group) == w.seq - w.residual
    ky, vy = cache.dequantize()
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for l in range(0, w.layers, 3):
        k, v = hosts[l]
        sample_keys(np.ascontiguousarray(k[:, :n]), host_u32(cache.k_codes[l]),
                    host_f32_bits(cache.k_scale[l]), host_f32_bits(cache.k_zero[l]),
                    host_u16(ky[l]), w.group, w.bits, 200, rng)
        sample_values(np.ascontiguousarray(v[:, :n]), host_u32(cache.v_codes[l]),
                      host_f32_bits(cache.v_scale[l]), host_f32_bits(cache.v_zero[l]),
                      host_u16(vy[l]), w.group, w.bits, 200, rng)
    # the last layer complete, every group and element: its tiles are among the
    # last each grid takes (late grid-stride iterations, the ring's last rows)
    l = w.layers - 1
    k, v = (np.ascontiguousarray(a[:, :n]) for a in hosts[l])
    oc, os_, oz = O.quantize_keys(k, w.group, w.bits)
    Wd = 32 // w.bits
    assert_same("last layer key codes", host_u32(cache.k_codes[l])[:, :n // Wd], oc)
    assert_same("last layer key scale", host_f32_bits(cache.k_scale[l])[:, :n // w.group],
                bits32(os_))
    assert_same("last layer key zero", host_f32_bits(cache.k_zero[l])[:, :n // w.group],
                bits32(oz))
    assert_same("last layer key recon", host_u16(ky[l]),
                O.dequantize_keys(oc, os_, oz, n, w.group, w.bits))
    oc, os_, oz = O.quantize_values(v, w.group, w.bits)
    assert_same("last layer value codes", host_u32(cache.v_codes[l])[:, :n], oc)
    assert_same("last layer value scale", host_f32_bits(cache.v_scale[l])[:, :n], bits32(os_))
    assert_same("last layer value zero", host_f32_bits(cache.v_zero[l])[:, :n], bits32(oz))
    assert_same("last layer value recon", host_u16(vy[l]),
                O.dequantize_values(oc, os_, oz, w.group, w.bits))


@pytest.mark.slow
def test_large_store_sweep_full_size_sampled(key_quantizer):
    w = W.CONFIGS["large_store_sweep"]
    k = W.generate(w, 0, "k")
    v = W.generate(w, 0, "v")
    kd, vd = to_dev(k), to_dev(v)
    rng = np.random.default_rng(6)
    last = w.bh - 1            # one complete bh slice per cell: the grid's last tiles
    kl, vl = np.ascontiguousarray(k[last:]), np.ascontiguousarray(v[last:])
    for bits in w.sweep_bits:
        for group in w.sweep_groups:
            c, s, z = K.kivi_quantize_keys(kd, group, bits)
            y = K.kivi_dequantize_keys(c, s, z, w.seq, group, bits)
            fy, fc, fs, fz = K.kivi_fakequant_keys(kd, group, bits)
            torch.cuda.synchronize()
            sample_keys(k, host_u32(c), host_f32_bits(s), host_f32_bits(z), host_u16(y),
                        group, bits, 60, rng)
            oc, os_, oz = O.quantize_keys(kl, group, bits)
            oy = O.dequantize_keys(oc, os_, oz, w.seq, group, bits)
            for name, got, want in (("key codes", host_u32(c[last:]), oc),
                                    ("key scale", host_f32_bits(s[last:]), bits32(os_)),
                                    ("key zero", host_f32_bits(z[last:]), bits32(oz)),
                                    ("key recon", host_u16(y[last:]), oy),
                                    ("fused key recon", host_u16(fy[last:]), oy),
                                    ("fused key codes", host_u32(fc[last:]), oc),
                                    ("fused key scale", host_f32_bits(fs[last:]), bits32(os_))):
                assert_same(f"{name} b{bits} g{group}", got, want)
            del c, s, z, y, fy, fc, fs, fz
            c, s, z = K.kivi_quantize_values(vd, group, bits)
            y = K.kivi_dequantize_values(c, s, z, group, bits)
            fy, fc, fs, fz = K.kivi_fakequant_values(vd, group, bits)
            torch.cuda.synchronize()
            sample_values(v, host_u32(c), host_f32_bits(s), host_f32_bits(z), host_u16(y),
                          group, bits, 60, rng)
            oc, os_, oz = O.quantize_values(vl, group, bits)
            oy = O.dequantize_values(oc, os_, oz, group, bits)
            for name, got, want in (("value codes", host_u32(c[last:]), oc),
                                    ("value scale", host_f32_bits(s[last:]), bits32(os_)),
                                    ("value zero", host_f32_bits(z[last:]), bits32(oz)),
                                    ("value recon", host_u16(y[last:]), oy),
                                    ("fused value recon", host_u16(fy[last:]), oy),
                                    ("fused value codes", host_u32(fc[last:]), oc),
                                    ("fused value zero", host_f32_bits(fz[last:]), bits32(oz))):
                assert_same(f"{name} b{bits} g{group}", got, want)
            del c, s, z, y, fy, fc, fs, fz


@pytest.mark.slow
def test_batched_decode_flushes_full_size_sampled(key_quantizer):
    """32 layers x 512 sequences: a store already holding 2048 tokens per
    sequence, a 64-token ring holding 32 fp16 tokens; each step appends 32
    tokens and the flush (one launch per kind over all layers) moves the 32
    oldest into the store at offset 2048 + 32 k."""
    w = W.CONFIGS["batched_decode"]
    steps = 3
    cap = w.store_prefill + w.new_per_step * (steps + 1)
    cache = K.KiviCache(w.layers, w.bh, w.head_dim, r_cap=2 * w.residual, cap=cap,
                        group=w.group, bits=w.bits, residual=w.residual)
    cache.reset(s_q=w.store_prefill, res_head=0, n_res=0)
    t_first = w.store_prefill

    def append(t0):
        for l in range(w.layers):
            k = W.generate(w, l, "k", tok0=t0, n_tok=w.new_per_step)
            v = W.generate(w, l, "v", tok0=t0, n_tok=w.new_per_step)
            cache.append(l, to_dev(k), to_dev(v))
        cache.advance(w.new_per_step)

    append(t_first)
    rng = np.random.default_rng(8)
    for step in range(steps):
        t_new = t_first + w.new_per_step * (step + 1)
        append(t_new)
        s_q0 = cache.s_q
        assert cache.flush() == w.new_per_step
        torch.cuda.synchronize()
        t_flushed = t_first + w.new_per_step * step
        for l in rng.choice(w.layers, 4, replace=False):
            k = W.generate(w, int(l), "k", tok0=t_flushed, n_tok=w.new_per_step)
            v = W.generate(w, int(l), "v", tok0=t_flushed, n_tok=w.new_per_step)
            sample_keys(k, host_u32(cache.k_codes[l]), host_f32_bits(cache.k_scale[l]),
                        host_f32_bits(cache.k_zero[l]), None, w.group, w.bits, 100, rng,
                        out_g0=s_q0 // w.group)
            sample_values(v, host_u32(cache.v_codes[l]), host_f32_bits(cache.v_scale[l]),
                          host_f32_bits(cache.v_zero[l]), None, w.group, w.bits, 100, rng,
                          out_r0=s_q0)
        # the last layer's flushed tokens complete (every sequence, head, channel)
        l = w.layers - 1
        n, G, Wd = w.new_per_step, w.group, 32 // w.bits
        k = W.generate(w, l, "k", tok0=t_flushed, n_tok=n)
        v = W.generate(w, l, "v", tok0=t_flushed, n_tok=n)
        oc, os_, oz = O.quantize_keys(k, G, w.bits)
        assert_same("key codes", host_u32(cache.k_codes[l])[:, s_q0 // Wd:(s_q0 + n) // Wd], oc)
        assert_same("key scale", host_f32_bits(cache.k_scale[l])[:, s_q0 // G:(s_q0 + n) // G],
                    bits32(os_))
        assert_same("key zero", host_f32_bits(cache.k_zero[l])[:, s_q0 // G:(s_q0 + n) // G],
                    bits32(oz))
        oc, os_, oz = O.quantize_values(v, G, w.bits)
        assert_same("value codes", host_u32(cache.v_codes[l])[:, s_q0:s_q0 + n], oc)
        assert_same("value scale", host_f32_bits(cache.v_scale[l])[:, s_q0:s_q0 + n], bits32(os_))
        assert_same("value zero", host_f32_bits(cache.v_zero[l])[:, s_q0:s_q0 + n], bits32(oz))
    assert cache.s_q == w.store_prefill + steps * w.new_per_step
