"""Bit-exact parity of the fused fake-quant path (quantize and dequantize in
one pass) with the CPU oracle, through the C ABI.

The expected reconstruction is the oracle's dequantization of the oracle's
quantization of the same input: the fused kernels must reproduce the
two-pass result bit for bit, together with the codes, scales and zeros when
those are requested.  The fused flush is checked on a multi-layer sequence
with ring wrap-around against the oracle's flush and against the library's
own batched dequantization of the store it wrote.
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


def _x(bh, s, d, seed, kind):
    w = W.custom(seed=seed, batch=1, kv_heads=bh, seq=s, head_dim=d,
                 keys=W.Dist(W.NORMAL, 1.0, n_outliers=min(4, d), outlier_mult=15.0))
    return W.generate(w, 0, kind)


def check_fq_keys(x: np.ndarray, group: int, bits: int) -> None:
    s = x.shape[1]
    oc, os_, oz = O.quantize_keys(x, group, bits)
    oy = O.dequantize_keys(oc, os_, oz, s, group, bits)
    xd = to_dev(x)
    y, c, sc, ze = K.kivi_fakequant_keys(xd, group, bits)
    y2, c2, _, _ = K.kivi_fakequant_keys(xd, group, bits, store=False)
    torch.cuda.synchronize()
    assert c2 is None
    assert_same("fused key recon", host_u16(y), oy)
    assert_same("fused key recon (no store)", host_u16(y2), oy)
    assert_same("fused key codes", host_u32(c), oc)
    assert_same("fused key scale", host_f32_bits(sc), bits32(os_))
    assert_same("fused key zero", host_f32_bits(ze), bits32(oz))


def check_fq_values(x: np.ndarray, group: int, bits: int) -> None:
    oc, os_, oz = O.quantize_values(x, group, bits)
    oy = O.dequantize_values(oc, os_, oz, group, bits)
    xd = to_dev(x)
    y, c, sc, ze = K.kivi_fakequant_values(xd, group, bits)
    y2, c2, _, _ = K.kivi_fakequant_values(xd, group, bits, store=False)
    torch.cuda.synchronize()
    assert c2 is None
    assert_same("fused value recon", host_u16(y), oy)
    assert_same("fused value recon (no store)", host_u16(y2), oy)
    assert_same("fused value codes", host_u32(c), oc)
    assert_same("fused value scale", host_f32_bits(sc), bits32(os_))
    assert_same("fused value zero", host_f32_bits(ze), bits32(oz))


@pytest.mark.parametrize("bits,group", COMBOS)
def test_fakequant_keys_several_tiles_ragged_tail(bits, group):
    check_fq_keys(_x(3, 3 * group + 5, 128, 5000 + bits * group, "k"), group, bits)


@pytest.mark.parametrize("bits,group", COMBOS)
def test_fakequant_values_several_rows(bits, group):
    check_fq_values(_x(3, 77, 128, 6000 + bits * group, "v"), group, bits)


@pytest.mark.parametrize("shape", [
    (1, 1, 128, 32, 2), (2, 5, 64, 64, 4), (1, 200, 8, 32, 2), (2, 100, 40, 64, 8),
    (1, 129, 256, 128, 2), (5, 31, 128, 32, 2), (2, 300, 16, 128, 8),
], ids=str)
def test_fakequant_keys_odd_shapes(shape):
    bh, s, d, g, b = shape
    check_fq_keys(_x(bh, s, d, 7000 + s + d, "k"), g, b)


@pytest.mark.parametrize("shape", [
    (1, 1, 32, 32, 2), (2, 50, 96, 32, 4), (1, 33, 256, 128, 8), (7, 3, 128, 128, 4),
    (3, 45, 64, 64, 2),
], ids=str)
def test_fakequant_values_odd_shapes(shape):
    bh, s, d, g, b = shape
    check_fq_values(_x(bh, s, d, 8000 + s + d, "v"), g, b)


@pytest.mark.parametrize("bits,group", COMBOS)
def test_fakequant_degenerate_and_tie_groups(bits, group):
    rng = np.random.default_rng(bits * 13 + group)
    bh, d = 2, 64
    blocks = [hard_block(rng, group, d) for _ in range(bh * 3)]
    x = np.stack([np.concatenate(blocks[3 * b:3 * b + 3], axis=0) for b in range(bh)])
    check_fq_keys(x.astype(np.float16).view(np.uint16), group, bits)
    s, d = 40, 2 * group
    x = np.stack([np.concatenate([hard_block(rng, group, s).T for _ in range(d // group)], axis=1)
                  for _ in range(bh)])
    check_fq_values(x.astype(np.float16).view(np.uint16), group, bits)


def test_fakequant_strided_output_leaves_padding():
    bh, s, d, g, b = 3, 70, 128, 32, 4
    x = _x(bh, s, d, 91, "k")
    y = torch.zeros((bh, s + 9, d), dtype=torch.float16, device="cuda")
    K.kivi_fakequant_keys(to_dev(x), g, b, y=y[:, :s], store=False)
    yv = torch.zeros((bh, s + 9, d), dtype=torch.float16, device="cuda")
    K.kivi_fakequant_values(to_dev(x), g, b, y=yv[:, :s], store=False)
    torch.cuda.synchronize()
    oc, os_, oz = O.quantize_keys(x, g, b)
    assert_same("recon", host_u16(y[:, :s]), O.dequantize_keys(oc, os_, oz, s, g, b))
    assert not host_u16(y[:, s:]).any()           # rows past s (ragged padding) untouched
    oc, os_, oz = O.quantize_values(x, g, b)
    assert_same("recon", host_u16(yv[:, :s]), O.dequantize_values(oc, os_, oz, g, b))
    assert not host_u16(yv[:, s:]).any()


def test_fakequant_partial_store_arguments_rejected():
    x = torch.zeros((1, 32, 128), dtype=torch.float16, device="cuda")
    y = torch.zeros_like(x)
    codes = torch.zeros((1, 2, 128), dtype=torch.int32, device="cuda")
    L = K.lib()
    rc = L.kivi_fakequant_keys(x.data_ptr(), 1, 32, 128, 32 * 128, 32, 2, y.data_ptr(),
                               32 * 128, codes.data_ptr(), 256, None, None, 128, None)
    assert rc == K.KIVI_ERR_INVAL
    torch.cuda.synchronize()
    assert not host_u16(y).any()


@pytest.mark.parametrize("bits,group,residual,store", [
    (2, 32, 32, True), (4, 64, 64, True), (8, 128, 32, True), (2, 64, 64, False)])
def test_fused_flush_sequence_with_ring_wrap(bits, group, residual, store):
    layers, bh, d = 3, 4, 128
    r_cap = 3 * group + (residual // group + 1) * group
    cap = 16 * group
    total = 14 * group
    w = W.custom(seed=80 + bits + group, batch=1, kv_heads=bh, seq=total, head_dim=d)
    K_all = [W.generate(w, l, "k") for l in range(layers)]
    V_all = [W.generate(w, l, "v") for l in range(layers)]
    cache = K.KiviCache(layers, bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                        residual=residual, recon=True, store=store)
    ring_k = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    ring_v = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    stores = [O.Store(bh, d, cap, group, bits) for _ in range(layers)]
    s_q = head = n_res = pos = 0
    rng = np.random.default_rng(bits + 3 * group)
    while pos < total:
        n_new = int(min(total - pos, rng.integers(1, 2 * group), r_cap - n_res))
        rows = (head + n_res + np.arange(n_new)) % r_cap
        for l in range(layers):
            ring_k[l][:, rows] = K_all[l][:, pos:pos + n_new]
            ring_v[l][:, rows] = V_all[l][:, pos:pos + n_new]
            cache.append(l, to_dev(K_all[l][:, pos:pos + n_new]),
                         to_dev(V_all[l][:, pos:pos + n_new]))
        cache.advance(n_new)
        n_res += n_new
        pos += n_new
        n_gpu = cache.flush_fakequant()
        for l in range(layers):
            n, s_q2, head2, n_res2 = O.flush(ring_k[l], ring_v[l], stores[l], residual,
                                              s_q, head, n_res)
        s_q, head, n_res = s_q2, head2, n_res2
        assert n_gpu == n and (cache.s_q, cache.res_head, cache.n_res) == (s_q, head, n_res)
    assert s_q >= 8 * group
    torch.cuda.synchronize()
    if store:
        ky, vy = cache.dequantize()
        torch.cuda.synchronize()
    for l in range(layers):
        st = stores[l]
        want_k = O.dequantize_keys(st.k_codes[:, :s_q // (32 // bits)], st.k_scale[:, :s_q // group],
                                   st.k_zero[:, :s_q // group], s_q, group, bits)
        want_v = O.dequantize_values(st.v_codes[:, :s_q], st.v_scale[:, :s_q],
                                     st.v_zero[:, :s_q], group, bits)
        assert_same("fused key recon", host_u16(cache.k_hat[l][:, :s_q]), want_k)
        assert_same("fused value recon", host_u16(cache.v_hat[l][:, :s_q]), want_v)
        assert not host_u16(cache.k_hat[l][:, s_q:]).any()
        assert not host_u16(cache.v_hat[l][:, s_q:]).any()
        if store:
            assert_same("store key codes", host_u32(cache.k_codes[l]), st.k_codes)
            assert_same("store key scale", host_f32_bits(cache.k_scale[l]), bits32(st.k_scale))
            assert_same("store value codes", host_u32(cache.v_codes[l]), st.v_codes)
            assert_same("store value zero", host_f32_bits(cache.v_zero[l]), bits32(st.v_zero))
            assert torch.equal(ky[l], cache.k_hat[l][:, :s_q])
            assert torch.equal(vy[l], cache.v_hat[l][:, :s_q])


@pytest.mark.slow
def test_fused_prefill_flush_full_size_sampled():
    """The 28-layer, 8-head, 4096-token prefill flush in its fused form: one
    launch per tensor kind writes the store and the fp16 reconstruction."""
    w = W.CONFIGS["llama3_2_3b_prefill"]
    cache = K.KiviCache(w.layers, w.bh, w.head_dim, r_cap=w.seq, cap=w.seq, group=w.group,
                        bits=w.bits, residual=w.residual, recon=True)
    hosts = []
    for l in range(w.layers):
        k = W.generate(w, l, "k")
        v = W.generate(w, l, "v")
        cache.k_res[l].copy_(to_dev(k))
        cache.v_res[l].copy_(to_dev(v))
        hosts.append((k, v))
    cache.advance(w.seq)
    n = cache.flush_fakequant()
    assert n == w.seq - w.residual
    torch.cuda.synchronize()
    rng = np.random.default_rng(15)
    for l in range(0, w.layers, 4):
        k, v = hosts[l]
        sample_keys(np.ascontiguousarray(k[:, :n]), host_u32(cache.k_codes[l]),
                    host_f32_bits(cache.k_scale[l]), host_f32_bits(cache.k_zero[l]),
                    host_u16(cache.k_hat[l]), w.group, w.bits, 200, rng)
        sample_values(np.ascontiguousarray(v[:, :n]), host_u32(cache.v_codes[l]),
                      host_f32_bits(cache.v_scale[l]), host_f32_bits(cache.v_zero[l]),
                      host_u16(cache.v_hat[l]), w.group, w.bits, 200, rng)
    ky, vy = cache.dequantize()
    torch.cuda.synchronize()
    for l in range(w.layers):
        assert torch.equal(ky[l], cache.k_hat[l][:, :n])
        assert torch.equal(vy[l], cache.v_hat[l][:, :n])
