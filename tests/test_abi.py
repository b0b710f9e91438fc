"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point declared in include/kivi.h, and its host-side logic (argument
validation, sizes, flush-size rule, empty calls) behaves as documented --
none of these paths makes a CUDA call."""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest

import kv_cache_quantization_kivi_gb300 as K
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kivi.h")

FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kivi_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    L = K.lib()
    names = declared_functions()
    assert {"kivi_quantize_keys", "kivi_quantize_values", "kivi_dequantize_keys",
            "kivi_dequantize_values", "kivi_flush"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert L.kivi_abi_version() == 1


def test_library_is_the_in_tree_build():
    assert os.path.exists(K.library_path())
    assert os.path.commonpath([K.library_path(), ROOT]) == ROOT


def test_status_strings():
    L = K.lib()
    for s in range(5):
        assert L.kivi_status_string(s)
    assert L.kivi_last_cuda_error() == 0


def test_flush_size_rule_matches_oracle():
    L = K.lib()
    for n_res in list(range(0, 300, 7)) + [559, 2059, 8209]:
        for r, g in [(32, 32), (64, 64), (0, 32), (32, 128), (5, 64)]:
            assert L.kivi_flush_size(n_res, r, g) == O.flush_size(n_res, r, g)
    assert L.kivi_flush_size(-1, 32, 32) == -1
    assert L.kivi_flush_size(10, 32, 0) == -1


def test_code_word_counts():
    assert K.kivi_key_code_words(100, 128, 32, 2) == 128 // 16 * 128
    assert K.kivi_key_code_words(4096, 128, 64, 4) == 4096 // 8 * 128
    assert K.kivi_value_code_words(100, 128, 32, 8) == 100 * 32
    assert K.kivi_value_code_words(7, 64, 64, 2) == 7 * 4
    assert K.kivi_key_code_words(10, 128, 48, 2) == -1
    assert K.kivi_value_code_words(10, 128, 32, 3) == -1


def _qk(**kw):
    a = dict(x=FAKE, bh=2, s=64, d=128, xs=64 * 128, group=32, bits=2, codes=FAKE,
             cs=64 // 16 * 128, scale=FAKE, zero=FAKE, ss=2 * 128, stream=None)
    a.update(kw)
    return K.lib().kivi_quantize_keys(a["x"], a["bh"], a["s"], a["d"], a["xs"], a["group"],
                                      a["bits"], a["codes"], a["cs"], a["scale"], a["zero"],
                                      a["ss"], a["stream"])


def _qv(**kw):
    a = dict(x=FAKE, bh=2, s=10, d=128, xs=10 * 128, group=32, bits=2, codes=FAKE,
             cs=10 * 8, scale=FAKE, zero=FAKE, ss=10 * 4, stream=None)
    a.update(kw)
    return K.lib().kivi_quantize_values(a["x"], a["bh"], a["s"], a["d"], a["xs"], a["group"],
                                        a["bits"], a["codes"], a["cs"], a["scale"], a["zero"],
                                        a["ss"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(bits=3), 1), (dict(bits=16), 1), (dict(group=48), 1), (dict(group=8), 1),
    (dict(group=256), 1),
    (dict(d=100), 1), (dict(d=264), 1), (dict(d=0), 1), (dict(bh=-1), 1), (dict(s=-3), 1),
    (dict(x=None), 1), (dict(codes=None), 1), (dict(zero=None), 1),
    (dict(xs=64 * 128 - 8), 1), (dict(cs=100), 1), (dict(ss=128), 1),
    (dict(x=FAKE + 8), 2), (dict(codes=FAKE + 4), 2), (dict(scale=FAKE + 8), 2),
    (dict(xs=64 * 128 + 4), 2), (dict(cs=64 // 16 * 128 + 1), 2), (dict(ss=2 * 128 + 1), 2),
    (dict(bh=0, x=None), 0), (dict(s=0, codes=None), 0),
])
def test_quantize_keys_validation(kw, status):
    assert _qk(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(bits=5), 1), (dict(group=64, d=96), 1), (dict(d=16), 1), (dict(d=48), 1),
    (dict(group=16, d=48), 1), (dict(group=16, d=16), 1), (dict(group=8, d=64), 1),
    (dict(scale=None), 1), (dict(cs=10 * 8 - 1), 1), (dict(ss=10 * 4 - 1), 1),
    (dict(xs=10 * 128 + 4), 2), (dict(bits=4, cs=10 * 16 + 2), 2), (dict(zero=FAKE + 4), 2),
    (dict(bh=0), 0), (dict(s=0), 0),
])
def test_quantize_values_validation(kw, status):
    assert _qv(**kw) == status


def test_dequantize_validation():
    L = K.lib()
    # keys: y stride too small, then misaligned y
    assert L.kivi_dequantize_keys(FAKE, 512, FAKE, FAKE, 256, 2, 64, 128, 32, 2, FAKE,
                                  64 * 128 - 8, None) == 1
    assert L.kivi_dequantize_keys(FAKE, 512, FAKE, FAKE, 256, 2, 64, 128, 32, 2, FAKE + 2,
                                  64 * 128, None) == 2
    assert L.kivi_dequantize_keys(FAKE, 512, FAKE, FAKE, 256, 0, 64, 128, 32, 2, None,
                                  64 * 128, None) == 0
    assert L.kivi_dequantize_values(FAKE, 80, FAKE, FAKE, 40, 2, 10, 128, 32, 3, FAKE,
                                    1280, None) == 1
    assert L.kivi_dequantize_values(FAKE, 80, FAKE, FAKE, 40, 2, 0, 128, 32, 2, FAKE,
                                    1280, None) == 0


def _cache(**kw):
    c = K.kivi_cache(bh=4, d=128, r_cap=128, cap=256, group=32, bits=2, residual=32,
                     reserved=0, s_q=0, res_head=0, n_res=40)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _layers(n=2, **kw):
    arr = (K.kivi_layer * n)()
    for i in range(n):
        for f, _ in K.kivi_layer._fields_:
            setattr(arr[i], f, FAKE + 4096 * i)
        for f, v in kw.items():
            setattr(arr[i], f, v)
    return arr


def _flush(layers, n, cache):
    out = C.c_int64(-7)
    rc = K.lib().kivi_flush(layers, n, C.byref(cache), C.byref(out), None)
    return rc, out.value


def test_flush_nothing_to_move_launches_nothing():
    c = _cache(n_res=63)
    rc, n = _flush(_layers(), 2, c)
    assert (rc, n) == (0, 0) and (c.s_q, c.res_head, c.n_res) == (0, 0, 63)


@pytest.mark.parametrize("kw", [
    dict(bits=3), dict(group=8), dict(residual=-1), dict(reserved=1), dict(d=80),
    dict(r_cap=100), dict(cap=250), dict(s_q=16), dict(s_q=288), dict(res_head=16),
    dict(res_head=128), dict(n_res=129), dict(n_res=-1), dict(bh=-2),
])
def test_flush_rejects_bad_cache_state(kw):
    c = _cache(**kw)
    before = (c.s_q, c.res_head, c.n_res)
    rc, _ = _flush(_layers(), 2, c)
    assert rc == 1
    assert (c.s_q, c.res_head, c.n_res) == before


def test_flush_rejects_bad_layers():
    c = _cache(n_res=100)
    assert _flush(_layers(), 0, c)[0] == 1
    assert _flush(_layers(), K.KIVI_MAX_LAYERS + 1, c)[0] == 1
    assert _flush(_layers(v_zero=None), 2, c)[0] == 1
    assert _flush(_layers(k_scale=FAKE + 4), 2, c)[0] == 2


def test_flush_capacity_error_leaves_state():
    c = _cache(cap=64, s_q=32, n_res=128)    # would move 96 tokens into 32 free
    rc, _ = _flush(_layers(), 2, c)
    assert rc == 3
    assert (c.s_q, c.res_head, c.n_res) == (32, 0, 128)


def test_flush_with_no_sequences_advances_state_only():
    c = _cache(bh=0, n_res=100)
    rc, n = _flush(_layers(), 2, c)
    assert (rc, n) == (0, 64) and (c.s_q, c.res_head, c.n_res) == (64, 64, 36)


def test_dequantize_cache_empty_store_is_a_noop():
    c = _cache(s_q=0)
    ptrs = (C.c_void_p * 2)(FAKE, FAKE)
    assert K.lib().kivi_dequantize_cache(_layers(), 2, C.byref(c), ptrs, ptrs, None) == 0


def _fq(fn, **kw):
    a = dict(x=FAKE, bh=2, s=64, d=128, xs=64 * 128, group=32, bits=2, y=FAKE + 65536,
             ys=64 * 128, codes=FAKE, cs=64 // 16 * 128, scale=FAKE, zero=FAKE, ss=2 * 128,
             stream=None)
    a.update(kw)
    return getattr(K.lib(), fn)(a["x"], a["bh"], a["s"], a["d"], a["xs"], a["group"], a["bits"],
                                a["y"], a["ys"], a["codes"], a["cs"], a["scale"], a["zero"],
                                a["ss"], a["stream"])


@pytest.mark.parametrize("fn", ["kivi_fakequant_keys", "kivi_fakequant_values"])
@pytest.mark.parametrize("kw,status", [
    (dict(y=None), 1), (dict(x=None), 1), (dict(bits=3), 1), (dict(group=8), 1),
    (dict(codes=None), 1), (dict(scale=None), 1), (dict(codes=None, zero=None), 1),
    (dict(ys=64 * 128 - 8), 1), (dict(xs=64 * 128 - 8), 1),
    (dict(y=FAKE + 2), 2), (dict(ys=64 * 128 + 4), 2), (dict(codes=FAKE + 4), 2),
    (dict(bh=0, x=None, y=None), 0), (dict(s=0), 0),
    (dict(s=1 << 62), 1), (dict(bh=1 << 40), 1), (dict(bh=1 << 62, s=1 << 62), 1),
])
def test_fakequant_validation(fn, kw, status):
    assert _fq(fn, **kw) == status


@pytest.mark.parametrize("kw", [dict(s=1 << 62), dict(bh=1 << 40), dict(bh=1 << 62, s=1 << 62)])
def test_huge_sizes_rejected_without_overflow(kw):
    assert _qk(**kw) == 1
    assert _qv(**kw) == 1
    L = K.lib()
    a = dict(bh=2, s=64)
    a.update(kw)
    assert L.kivi_dequantize_keys(FAKE, 512, FAKE, FAKE, 256, a["bh"], a["s"], 128, 32, 2,
                                  FAKE, 64 * 128, None) == 1
    assert L.kivi_dequantize_values(FAKE, 80, FAKE, FAKE, 40, a["bh"], a["s"], 128, 32, 2,
                                    FAKE, 1280, None) == 1


def test_flush_rejects_huge_ring():
    c = _cache(r_cap=1 << 40, n_res=100)
    assert _flush(_layers(), 2, c)[0] == 1


def _flush_fq(layers, n, cache, k_hat, v_hat):
    out = C.c_int64(-7)
    rc = K.lib().kivi_flush_fakequant(layers, n, C.byref(cache), k_hat, v_hat, C.byref(out),
                                      None, None)
    return rc, out.value


def test_fused_flush_validation():
    hat = (C.c_void_p * 2)(FAKE + (1 << 20), FAKE + (2 << 20))
    c = _cache(n_res=63)          # nothing to move: validated, then no launch
    assert _flush_fq(_layers(), 2, c, hat, hat) == (0, 0)
    # store pointers may be all NULL for a tensor kind (reconstruction only)
    c = _cache(n_res=63)
    assert _flush_fq(_layers(k_codes=None, k_scale=None, k_zero=None), 2, c, hat, hat)[0] == 0
    assert _flush_fq(_layers(v_codes=None, v_scale=None, v_zero=None), 2, c, hat, hat)[0] == 0
    # ... but not partly, and never for the plain flush
    assert _flush_fq(_layers(k_codes=None), 2, c, hat, hat)[0] == 1
    assert _flush(_layers(k_codes=None, k_scale=None, k_zero=None), 2, c)[0] == 1
    assert _flush_fq(_layers(k_res=None), 2, c, hat, hat)[0] == 1
    # reconstruction arrays
    assert _flush_fq(_layers(), 2, c, None, hat)[0] == 1
    assert _flush_fq(_layers(), 2, c, (C.c_void_p * 2)(FAKE, None), hat)[0] == 1
    assert _flush_fq(_layers(), 2, c, (C.c_void_p * 2)(FAKE, FAKE + 8), hat)[0] == 2
    # capacity and state rules are those of the flush
    c = _cache(cap=64, s_q=32, n_res=128)
    assert _flush_fq(_layers(), 2, c, hat, hat)[0] == 3
    assert (c.s_q, c.res_head, c.n_res) == (32, 0, 128)
    c = _cache(bh=0, n_res=100)
    assert _flush_fq(_layers(), 2, c, hat, hat) == (0, 64)


def _attn(cache, layers=None, n=2, batch=2, h_q=8, scale=0.1, q=None, out=None, n_split=1,
          ws=None, ws_n=0):
    q = q if q is not None else (C.c_void_p * n)(*[FAKE + (1 << 24) * (i + 1) for i in range(n)])
    out = out if out is not None else (C.c_void_p * n)(*[FAKE + (1 << 28) * (i + 1)
                                                          for i in range(n)])
    return K.lib().kivi_decode_attention(layers if layers is not None else _layers(n), n,
                                         C.byref(cache), batch, h_q, scale, q, out, n_split, ws,
                                         ws_n, None)


def test_decode_attention_validation():
    # bh = 4: batch 2 -> h_kv 2; h_q 8 -> r = 4
    assert _attn(_cache(d=96)) == 1                         # head_dim 64, 128 or 256 only
    assert _attn(_cache(d=32)) == 1
    assert K.lib().kivi_decode_attention_workspace(C.byref(_cache(d=96)), 2, 2, 8, 2) == -1
    for d in (64, 256):                                      # partials of d + 2 floats
        assert K.lib().kivi_decode_attention_workspace(C.byref(_cache(d=d)), 2, 2, 8, 2) == \
            2 * 4 * 2 * 4 * (d + 2)
    assert _attn(_cache(), batch=3) == 1                    # bh % batch
    assert _attn(_cache(), h_q=7) == 1                      # h_q % h_kv
    assert _attn(_cache(), h_q=18) == 1                     # r = 9 > 8
    assert _attn(_cache(), n_split=0) == 1
    assert _attn(_cache(), n_split=65) == 1
    assert _attn(_cache(), n_split=2) == 1                  # no workspace
    need = K.lib().kivi_decode_attention_workspace(C.byref(_cache()), 2, 2, 8, 2)
    assert need == 2 * 4 * 2 * 4 * 130
    assert _attn(_cache(), n_split=2, ws=FAKE, ws_n=need - 1) == 1
    assert _attn(_cache(), n_split=2, ws=FAKE + 4, ws_n=need) == 2
    assert _attn(_cache(), q=(C.c_void_p * 2)(FAKE, None)) == 1
    assert _attn(_cache(), q=(C.c_void_p * 2)(FAKE, FAKE + 2)) == 2
    assert _attn(_cache(), scale=float("nan")) == 1
    assert _attn(_cache(s_q=0, n_res=0)) == 1               # nothing to attend to
    assert _attn(_cache(bh=0), batch=1) == 1                # bh 0: no sequence to map
    assert _attn(_cache(), layers=_layers(2, v_zero=None)) == 1
    assert K.lib().kivi_decode_attention_workspace(C.byref(_cache()), 2, 2, 8, 1) == 0
    assert K.lib().kivi_decode_attention_workspace(C.byref(_cache()), 2, 2, 9, 1) == -1
    assert K.lib().kivi_decode_attention_splits(C.byref(_cache()), 2, 2) >= 1


def test_selftest_wait_limits():
    assert K.lib().kivi_selftest_wait_timeout(0, None) == 1
    assert K.lib().kivi_selftest_wait_timeout(1_000_001, None) == 1


def test_device_fault_rejects_null():
    assert K.lib().kivi_device_fault(None) == 1


def test_decode_attention_noalloc_validation():
    L = K.lib()
    q = (C.c_void_p * 2)(FAKE + (1 << 24), FAKE + (2 << 24))
    out = (C.c_void_p * 2)(FAKE + (1 << 28), FAKE + (2 << 28))
    # workspace need 2 * 4096 * 64 * 8 * 130 floats > the fixed 2^24: refused before any CUDA call
    big = _cache(bh=4096, n_res=40)
    assert L.kivi_decode_attention_noalloc(_layers(2), 2, C.byref(big), 512, 64, 0.1, q, out, 64,
                                           None) == 3
    # argument errors keep their own status
    assert L.kivi_decode_attention_noalloc(_layers(2), 2, C.byref(_cache()), 3, 8, 0.1, q, out,
                                           2, None) == 1
    assert L.kivi_decode_attention_noalloc(_layers(2), 2, C.byref(_cache()), 2, 8, 0.1, q, out,
                                           0, None) == 1
    assert L.kivi_decode_attention_noalloc(_layers(2), 2, C.byref(_cache(bh=0)), 1, 8, 0.1, q,
                                           out, 2, None) == 1


def _sinks(n=2, **kw):
    arr = (K.kivi_sink_layer * n)()
    for i in range(n):
        for f, _ in K.kivi_sink_layer._fields_:
            setattr(arr[i], f, FAKE + (1 << 20) * (i + 1))
        for f, v in kw.items():
            setattr(arr[i], f, v)
    return arr


def test_sink_validation():
    L = K.lib()
    c = _cache(n_res=40)
    cfg = lambda **kw: K.kivi_sink_cfg(**{**dict(batch=2, k_top=5, sink_cap=8, reserved=0,  # noqa
                                                   reserved2=0), **kw})
    upd = lambda cc, s, cf, i0, n: L.kivi_sink_update(_layers(2), s, 2, C.byref(cc),  # noqa
                                                      C.byref(cf), i0, n, None)
    assert upd(c, _sinks(), cfg(batch=3), 0, 8) == 1            # bh % batch
    assert upd(c, _sinks(), cfg(k_top=65), 0, 8) == 1           # top-k beyond 64
    assert upd(c, _sinks(), cfg(k_top=-1), 0, 8) == 1
    assert upd(c, _sinks(), cfg(reserved=1), 0, 8) == 1
    assert upd(c, _sinks(mask=None), cfg(), 0, 8) == 1
    assert upd(c, _sinks(sink_k=FAKE + 4), cfg(), 0, 8) == 2
    assert upd(c, _sinks(), cfg(), 30, 11) == 1                 # past the residual
    assert upd(c, _sinks(), cfg(), 0, 0) == 0                   # nothing to score
    assert upd(c, _sinks(), cfg(k_top=0), 0, 8) == 0            # no top-k kept
    # launch sizes beyond 2^31 - 1 units are refused before any launch: 128
    # layers x 2^16 sequences x 2^10 ring rows of tokens to score, and 128 x
    # 2^16 sequence-heads x 2^10 sink slots x 4 pieces to restore
    upd128 = lambda cc, cf: L.kivi_sink_update(_layers(128), _sinks(128), 128,  # noqa
                                                C.byref(cc), C.byref(cf), 0, 8, None)
    big = _cache(bh=1 << 16, d=32, r_cap=1 << 10, cap=0, n_res=40)
    assert upd128(big, cfg(batch=1 << 16, sink_cap=0)) == 1
    mid = _cache(bh=1 << 10, d=32, r_cap=32, cap=0, n_res=32)
    assert upd128(mid, cfg(batch=1 << 10, sink_cap=1 << 14)) == 1
    out = C.c_int64(-1)
    c2 = _cache(n_res=63)                                       # nothing to flush
    assert L.kivi_flush_sink(_layers(2), _sinks(), 2, C.byref(c2), C.byref(cfg()),
                             C.byref(out), None) == 0 and out.value == 0
    c3 = _cache(cap=64, s_q=32, n_res=128)
    assert L.kivi_flush_sink(_layers(2), _sinks(), 2, C.byref(c3), C.byref(cfg()),
                             C.byref(out), None) == 3
    assert (c3.s_q, c3.n_res) == (32, 128)
    ptrs = (C.c_void_p * 2)(FAKE, FAKE)
    assert L.kivi_sink_restore(_sinks(), 2, C.byref(_cache(s_q=0)), C.byref(cfg()), ptrs, ptrs,
                               None) == 0
    assert L.kivi_sink_restore(_sinks(), 2, C.byref(_cache(s_q=32)), C.byref(cfg()),
                               (C.c_void_p * 2)(FAKE, None), ptrs, None) == 1


def test_decode_attention_sinks_validation():
    L = K.lib()
    q = (C.c_void_p * 2)(FAKE + (1 << 24), FAKE + (2 << 24))
    out = (C.c_void_p * 2)(FAKE + (1 << 28), FAKE + (2 << 28))
    cfg = lambda **kw: K.kivi_sink_cfg(**{**dict(batch=2, k_top=5, sink_cap=8, reserved=0,  # noqa
                                                   reserved2=0), **kw})
    call = lambda c, s, cf, batch=2, n_split=1: L.kivi_decode_attention_sinks(  # noqa
        _layers(2), s, 2, C.byref(c), C.byref(cf), batch, 8, 0.1, q, out, n_split, None, 0, None)
    assert call(_cache(), _sinks(), cfg(batch=1)) == 1          # cfg batch != batch
    assert call(_cache(), _sinks(sink_pos=None), cfg()) == 1
    assert call(_cache(), _sinks(sink_k=FAKE + 4), cfg()) == 2
    assert call(_cache(), _sinks(), cfg(reserved=1)) == 1
    assert call(_cache(d=96), _sinks(), cfg()) == 1             # head_dim 64, 128 or 256 only
    assert call(_cache(), _sinks(), cfg(), n_split=2) == 1      # no workspace
    assert L.kivi_decode_attention_sinks(_layers(2), None, 2, C.byref(_cache()), C.byref(cfg()),
                                         2, 8, 0.1, q, out, 1, None, 0, None) == 1


def _append(layers, n_layers, cache, n, stride=None, k_new=FAKE, v_new=FAKE + 65536):
    kp = (C.c_void_p * max(n_layers, 1))(*([k_new] * max(n_layers, 1)))
    vp = (C.c_void_p * max(n_layers, 1))(*([v_new] * max(n_layers, 1)))
    stride = n * int(cache.d) if stride is None else stride
    return K.lib().kivi_append(layers, n_layers, C.byref(cache), kp, vp, stride, n, None)


def test_append_validation_leaves_state():
    """Argument errors of kivi_append launch nothing and leave n_res alone."""
    cases = [
        (dict(n_res=100), dict(n=40), 3),                 # 140 tokens in a 128-row ring
        (dict(n_res=0), dict(n=-1), 1),
        (dict(n_res=0), dict(n=8, stride=8 * 128 - 8), 1),   # stride below n * d
        (dict(n_res=0), dict(n=8, stride=8 * 128 + 4), 2),   # stride not 16-byte aligned
        (dict(n_res=0), dict(n=8, k_new=FAKE + 8), 2),
        (dict(n_res=0), dict(n=8, v_new=0), 1),
        (dict(n_res=0, res_head=128), dict(n=8), 1),       # head outside the ring
    ]
    for ckw, akw, status in cases:
        c = _cache(**ckw)
        before = (c.s_q, c.res_head, c.n_res)
        assert _append(_layers(), 2, c, **akw) == status, (ckw, akw)
        assert (c.s_q, c.res_head, c.n_res) == before


def test_append_of_nothing_advances_nothing():
    c = _cache(n_res=5)
    assert _append(_layers(), 2, c, 0) == 0 and c.n_res == 5
    c = _cache(bh=0, n_res=5)                              # no sequences: the count advances
    assert _append(_layers(), 2, c, 40) == 0 and c.n_res == 45


def test_append_accepts_layers_without_store():
    c = _cache(bh=0, n_res=0)
    L = _layers(k_codes=None, k_scale=None, k_zero=None, v_codes=None, v_scale=None,
                v_zero=None)
    assert _append(L, 2, c, 16) == 0 and c.n_res == 16


def _append_flush(layers, n_layers, cache, n, stride=None, events=None):
    kp = (C.c_void_p * n_layers)(*([FAKE] * n_layers))
    vp = (C.c_void_p * n_layers)(*([FAKE + 65536] * n_layers))
    stride = n * int(cache.d) if stride is None else stride
    out = C.c_int64(-7)
    rc = K.lib().kivi_append_flush(layers, n_layers, C.byref(cache), kp, vp, stride, n,
                                   C.byref(out), None, events)
    return rc, out.value


def test_append_flush_checks_both_steps_before_launching():
    """A flush that would overrun the store is refused before the append
    launches: the state (residual count included) is unchanged."""
    c = _cache(cap=64, s_q=32, n_res=40)      # 40 + 60 tokens -> flush of 64 into 32 free
    assert _append_flush(_layers(), 2, c, 60)[0] == 3
    assert (c.s_q, c.res_head, c.n_res) == (32, 0, 40)
    c = _cache(n_res=100)
    assert _append_flush(_layers(), 2, c, 40)[0] == 3          # ring overflow
    assert c.n_res == 100
    c = _cache(n_res=0)
    assert _append_flush(_layers(v_codes=None, v_scale=None, v_zero=None), 2, c, 8)[0] == 1
    assert _append_flush(_layers(), 2, c, 8, stride=8 * 128 + 4)[0] == 2


def test_append_flush_without_sequences_advances_both_steps():
    c = _cache(bh=0, n_res=32)
    rc, n = _append_flush(_layers(), 2, c, 64)                 # 96 in the residual -> flush 64
    assert (rc, n) == (0, 64) and (c.s_q, c.res_head, c.n_res) == (64, 64, 32)
