"""The residual ring's append (``kivi_append``) on the GPU against the
oracle's append, bit for bit: the rings of every layer after sequences of
appends that wrap the ring mid-chunk, interleaved with flushes whose store
must equal the oracle's, with contiguous and strided new-token tensors, at
several head dims and group sizes."""
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


def run_sequence(layers, bh, d, group, bits, r_cap, chunks, strided, seed, fused=False):
    cap = (sum(chunks) // group + 1) * group
    cache = K.KiviCache(layers, bh, d, r_cap=r_cap, cap=cap, group=group, bits=bits,
                        residual=group)
    w = W.custom(seed=seed, batch=1, kv_heads=bh, seq=sum(chunks), head_dim=d)
    rings = [(np.zeros((bh, r_cap, d), np.uint16), np.zeros((bh, r_cap, d), np.uint16))
             for _ in range(layers)]
    stores = [O.Store(bh, d, cap, group, bits) for _ in range(layers)]
    s_q = head = n_res = pos = 0
    wrapped = False
    for n in chunks:
        ks = [W.generate(w, l, "k", tok0=pos, n_tok=n) for l in range(layers)]
        vs = [W.generate(w, l, "v", tok0=pos, n_tok=n) for l in range(layers)]
        if strided:
            # the new tokens as a view of a wider tensor: bh stride (n + 8) * d
            kd = [torch.zeros((bh, n + 8, d), dtype=torch.float16, device="cuda")
                  for _ in range(layers)]
            vd = [torch.zeros((bh, n + 8, d), dtype=torch.float16, device="cuda")
                  for _ in range(layers)]
            for l in range(layers):
                kd[l][:, 3:3 + n] = to_dev(ks[l])
                vd[l][:, 3:3 + n] = to_dev(vs[l])
            kd = [t[:, 3:3 + n] for t in kd]
            vd = [t[:, 3:3 + n] for t in vd]
        else:
            kd = [to_dev(x) for x in ks]
            vd = [to_dev(x) for x in vs]
        wrapped |= (head + n_res) % r_cap + n > r_cap
        n_res2 = n_res
        for l in range(layers):
            n_res2 = O.append(rings[l][0], rings[l][1], head, n_res, ks[l], vs[l])
        if fused:
            # append and flush in one call (the flush's launches overlap the
            # append's tail when the flushed rows were in the ring before it)
            n_gpu = cache.append_flush(kd, vd)
        else:
            cache.append_all(kd, vd)
            assert cache.n_res == n_res2
            for l in range(layers):
                assert_same(f"key ring {l}", host_u16(cache.k_res[l]), rings[l][0])
                assert_same(f"value ring {l}", host_u16(cache.v_res[l]), rings[l][1])
            n_gpu = cache.flush()
        n_res = n_res2
        for l in range(layers):
            n_o, s_q2, head2, n_res2 = O.flush(rings[l][0], rings[l][1], stores[l], group,
                                               s_q, head, n_res)
        assert n_gpu == n_o
        s_q, head, n_res = s_q2, head2, n_res2
        assert (cache.s_q, cache.res_head, cache.n_res) == (s_q, head, n_res)
        pos += n
    torch.cuda.synchronize()
    for l in range(layers):
        st = stores[l]
        assert_same("key codes", host_u32(cache.k_codes[l]), st.k_codes)
        assert_same("key scale", host_f32_bits(cache.k_scale[l]), bits32(st.k_scale))
        assert_same("key zero", host_f32_bits(cache.k_zero[l]), bits32(st.k_zero))
        assert_same("value codes", host_u32(cache.v_codes[l]), st.v_codes)
        assert_same("value scale", host_f32_bits(cache.v_scale[l]), bits32(st.v_scale))
        assert_same("value zero", host_f32_bits(cache.v_zero[l]), bits32(st.v_zero))
    return wrapped, s_q


@pytest.mark.parametrize("bits,group,d,strided", [(2, 32, 128, False), (4, 64, 128, True),
                                                  (8, 16, 64, False), (2, 128, 256, True),
                                                  (4, 32, 96, False)])
def test_append_sequence_matches_oracle(bits, group, d, strided):
    r_cap = 4 * group
    rng = np.random.default_rng(bits * 100 + group + d)
    chunks = [3 * group]
    n_res = 3 * group
    while sum(chunks) < 12 * group:
        n_res -= O.flush_size(n_res, group, group)
        n = int(rng.integers(1, r_cap - n_res + 1))
        chunks.append(n)
        n_res += n
    wrapped, s_q = run_sequence(3, 5, d, group, bits, r_cap, chunks, strided,
                                seed=300 + bits + group)
    assert wrapped and s_q >= 8 * group


def test_decode_step_shape():
    """The decode benchmark's pattern: a 2R-row ring, R new tokens per step
    flushed one step later, 40 steps."""
    _, s_q = run_sequence(2, 16, 128, 32, 2, 64, [32] * 40, False, seed=311)
    assert s_q == 32 * 39          # the ring's head went round 20 times


@pytest.mark.parametrize("bits,group,r_groups", [(2, 32, 3), (4, 64, 4), (8, 16, 5)])
def test_append_flush_matches_oracle(bits, group, r_groups):
    """kivi_append_flush over decode-like steps (the flushed rows precede the
    appended ones: overlapped launches) and prefill-like chunks (some
    appended tokens flushed at once: the flush waits for the append)."""
    r_cap = r_groups * group
    rng = np.random.default_rng(bits + group)
    chunks, n_res, kinds = [], 0, set()
    while (len(chunks) < 14 or not {True, False} <= kinds) and len(chunks) < 200:
        room = r_cap - n_res
        n = int(rng.choice([group, room, 1 + int(rng.integers(room))]))
        f = O.flush_size(n_res + n, group, group)
        kinds.add(f <= n_res if f > 0 else None)
        chunks.append(n)
        n_res += n - f
    assert True in kinds and False in kinds
    _, s_q = run_sequence(2, 6, 128, group, bits, r_cap, chunks, False, seed=400 + bits + group,
                          fused=True)
    assert s_q >= 3 * group
