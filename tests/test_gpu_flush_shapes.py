"""The flush (plain and fused) at head dims other than 128: the generic
kernel instances (head_dim a runtime value) against the oracle's flush, over
a sequence of appends with ring wrap-around, several layers and every code
width."""
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


@pytest.mark.parametrize("d,bits,group,fused", [
    (64, 2, 32, False), (64, 4, 64, True), (256, 8, 32, False), (256, 2, 128, True),
    (96, 4, 32, True), (192, 2, 64, False), (256, 4, 64, False), (64, 8, 64, True),
    (64, 4, 16, True), (256, 2, 16, False), (96, 8, 16, True), (32, 2, 16, False),
])
def test_flush_sequence_other_head_dims(d, bits, group, fused):
    layers, bh, residual = 2, 3, group
    r_cap = 4 * group
    cap = 10 * group
    w = W.custom(seed=500 + d + bits, batch=1, kv_heads=bh, seq=cap + r_cap, head_dim=d)
    cache = K.KiviCache(layers, bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                        residual=residual, recon=fused)
    ring_k = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    ring_v = [np.zeros((bh, r_cap, d), np.uint16) for _ in range(layers)]
    stores = [O.Store(bh, d, cap, group, bits) for _ in range(layers)]
    s_q = head = n_res = pos = 0
    rng = np.random.default_rng(d + bits)
    while s_q + n_res < 9 * group:
        n_new = int(min(rng.integers(1, 2 * group), r_cap - n_res))
        rows = (head + n_res + np.arange(n_new)) % r_cap
        for l in range(layers):
            k = W.generate(w, l, "k", tok0=pos, n_tok=n_new)
            v = W.generate(w, l, "v", tok0=pos, n_tok=n_new)
            ring_k[l][:, rows] = k
            ring_v[l][:, rows] = v
            cache.append(l, to_dev(k), to_dev(v))
        cache.advance(n_new)
        n_res += n_new
        pos += n_new
        n_gpu = cache.flush_fakequant() if fused else cache.flush()
        for l in range(layers):
            n, s_q2, head2, n_res2 = O.flush(ring_k[l], ring_v[l], stores[l], residual, s_q,
                                              head, n_res)
        s_q, head, n_res = s_q2, head2, n_res2
        assert n_gpu == n and (cache.s_q, cache.res_head, cache.n_res) == (s_q, head, n_res)
    torch.cuda.synchronize()
    assert s_q >= 5 * group
    ky, vy = cache.dequantize()
    torch.cuda.synchronize()
    for l in range(layers):
        st = stores[l]
        assert_same("key codes", host_u32(cache.k_codes[l]), st.k_codes)
        assert_same("key scale", host_f32_bits(cache.k_scale[l]), bits32(st.k_scale))
        assert_same("key zero", host_f32_bits(cache.k_zero[l]), bits32(st.k_zero))
        assert_same("value codes", host_u32(cache.v_codes[l]), st.v_codes)
        assert_same("value scale", host_f32_bits(cache.v_scale[l]), bits32(st.v_scale))
        assert_same("value zero", host_f32_bits(cache.v_zero[l]), bits32(st.v_zero))
        kref, vref = O.cache_kv(st, s_q, ring_k[l], ring_v[l], head, 0)
        assert_same("key recon", host_u16(ky[l]), kref)
        assert_same("value recon", host_u16(vy[l]), vref)
        if fused:
            assert_same("fused key recon", host_u16(cache.k_hat[l][:, :s_q]), kref)
            assert_same("fused value recon", host_u16(cache.v_hat[l][:, :s_q]), vref)
