"""ctypes wrapper around the C oracle (``kivi_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the product package never
imports this module and shares no code with it.

The oracle is built from source with the host C compiler the first time it is
needed (or by :func:`build`), into ``oracle/_build/``.  fp16 tensors are passed
as ``numpy.uint16`` arrays holding the IEEE binary16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_HDR = os.path.join(_HERE, "kivi_oracle.h")
_LIB = os.path.join(_HERE, "_build", "libkivi_oracle.so")
# -ffp-contract=off: no fused multiply-add; -fno-fast-math: IEEE semantics,
# no flush-to-zero, no reassociation.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i64 = C.c_int64
_i64p = C.POINTER(C.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or stale."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc, *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # KIVI_ORACLE_LIB: a library built elsewhere from a copy of this
            # source (the planted-mistake test loads mutated builds this way)
            path = os.environ.get("KIVI_ORACLE_LIB") or build()
            L = C.CDLL(path)
            L.kivi_oracle_half_to_float.argtypes = [C.c_uint16]
            L.kivi_oracle_half_to_float.restype = C.c_float
            L.kivi_oracle_float_to_half.argtypes = [C.c_float]
            L.kivi_oracle_float_to_half.restype = C.c_uint16
            L.kivi_oracle_halves_to_floats.argtypes = [_u16p, _f32p, _i64]
            L.kivi_oracle_halves_to_floats.restype = None
            L.kivi_oracle_floats_to_halves.argtypes = [_f32p, _u16p, _i64]
            L.kivi_oracle_floats_to_halves.restype = None
            L.kivi_oracle_group_params.argtypes = [_f32p, _i64, C.c_int,
                                                   C.POINTER(C.c_float), C.POINTER(C.c_float)]
            L.kivi_oracle_group_params.restype = C.c_int
            L.kivi_oracle_code.argtypes = [C.c_float, C.c_float, C.c_float, C.c_int]
            L.kivi_oracle_code.restype = C.c_uint32
            L.kivi_oracle_recon.argtypes = [C.c_uint32, C.c_float, C.c_float]
            L.kivi_oracle_recon.restype = C.c_uint16
            for name in ("kivi_oracle_quantize_keys", "kivi_oracle_quantize_values"):
                f = getattr(L, name)
                f.argtypes = [_u16p, _i64, _i64, _i64, C.c_int, C.c_int, _u32p, _f32p, _f32p]
                f.restype = C.c_int
            for name in ("kivi_oracle_dequantize_keys", "kivi_oracle_dequantize_values"):
                f = getattr(L, name)
                f.argtypes = [_u32p, _f32p, _f32p, _i64, _i64, _i64, C.c_int, C.c_int, _u16p]
                f.restype = C.c_int
            L.kivi_oracle_key_group.argtypes = [_u16p, _i64, _i64, _i64, _i64, C.c_int, C.c_int,
                                                _u32p, C.POINTER(C.c_float), C.POINTER(C.c_float)]
            L.kivi_oracle_key_group.restype = C.c_int
            L.kivi_oracle_value_row.argtypes = [_u16p, _i64, C.c_int, C.c_int, _u32p, _f32p, _f32p]
            L.kivi_oracle_value_row.restype = C.c_int
            L.kivi_oracle_flush_size.argtypes = [_i64, C.c_int, C.c_int]
            L.kivi_oracle_flush_size.restype = _i64
            L.kivi_oracle_flush.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _i64,
                                            C.c_int, C.c_int, C.c_int,
                                            _u32p, _f32p, _f32p, _u32p, _f32p, _f32p,
                                            _i64p, _i64p, _i64p]
            L.kivi_oracle_flush.restype = _i64
            L.kivi_oracle_append.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _i64, _i64p,
                                             _u16p, _u16p, _i64]
            L.kivi_oracle_append.restype = C.c_int
            L.kivi_oracle_attention.argtypes = [_u16p, _i64, _u16p, _u16p, _i64, _i64,
                                                C.c_double, _f64p]
            L.kivi_oracle_attention.restype = C.c_int
            _i64a = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
            L.kivi_oracle_sink_scores.argtypes = [_u16p, _i64, _i64, _i64, _i64, _i64, _f32p]
            L.kivi_oracle_sink_scores.restype = C.c_int
            L.kivi_oracle_sink_topk.argtypes = [_i64, _i64a, _f32p, _i64p, _f32p, _i64, _i64]
            L.kivi_oracle_sink_topk.restype = C.c_int
            L.kivi_oracle_flush_sink.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _i64, _i64,
                                                 C.c_int, C.c_int, C.c_int, _u32p, _f32p, _f32p,
                                                 _u32p, _f32p, _f32p, _i64p, _i64p, _i64p,
                                                 _i64, _i64a, _i64a, _i64, _i64a, _i64a,
                                                 _u16p, _u16p]
            L.kivi_oracle_flush_sink.restype = _i64
            L.kivi_oracle_sink_restore.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _i64, _i64,
                                                   _i64a, _i64a, _u16p, _u16p]
            L.kivi_oracle_sink_restore.restype = C.c_int
            _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def codes_per_word(bits: int) -> int:
    return 32 // bits


# --------------------------------------------------------------------------
# scalar / element-wise helpers
# --------------------------------------------------------------------------

def half_to_float(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().kivi_oracle_halves_to_floats(h.reshape(-1), out.reshape(-1), h.size)
    return out


def float_to_half(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().kivi_oracle_floats_to_halves(f.reshape(-1), out.reshape(-1), f.size)
    return out


def group_params(vals, bits: int):
    v = np.ascontiguousarray(vals, dtype=np.float32).reshape(-1)
    sc, ze = C.c_float(), C.c_float()
    _check(lib().kivi_oracle_group_params(v, v.size, bits, C.byref(sc), C.byref(ze)),
           "group_params")
    return np.float32(sc.value), np.float32(ze.value)


def code(x, scale, zero, bits: int) -> int:
    return int(lib().kivi_oracle_code(float(x), float(scale), float(zero), bits))


def recon(q: int, scale, zero) -> int:
    return int(lib().kivi_oracle_recon(int(q), float(scale), float(zero)))


# --------------------------------------------------------------------------
# full-tensor operations
# --------------------------------------------------------------------------

def quantize_keys(x: np.ndarray, group: int, bits: int):
    """x: uint16 [bh, s, d] -> (codes u32 [bh, ng*G/W, d], scale, zero f32 [bh, ng, d])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    bh, s, d = x.shape
    ng = -(-s // group)
    codes = np.zeros((bh, ng * group // codes_per_word(bits), d), np.uint32)
    scale = np.zeros((bh, ng, d), np.float32)
    zero = np.zeros((bh, ng, d), np.float32)
    _check(lib().kivi_oracle_quantize_keys(x, bh, s, d, group, bits, codes, scale, zero),
           "quantize_keys")
    return codes, scale, zero


def quantize_values(x: np.ndarray, group: int, bits: int):
    """x: uint16 [bh, s, d] -> (codes u32 [bh, s, d/W], scale, zero f32 [bh, s, d/G])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    bh, s, d = x.shape
    codes = np.zeros((bh, s, d // codes_per_word(bits)), np.uint32)
    scale = np.zeros((bh, s, d // group), np.float32)
    zero = np.zeros((bh, s, d // group), np.float32)
    _check(lib().kivi_oracle_quantize_values(x, bh, s, d, group, bits, codes, scale, zero),
           "quantize_values")
    return codes, scale, zero


def dequantize_keys(codes, scale, zero, s: int, group: int, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    zero = np.ascontiguousarray(zero, dtype=np.float32)
    bh, _, d = codes.shape
    y = np.zeros((bh, s, d), np.uint16)
    _check(lib().kivi_oracle_dequantize_keys(codes, scale, zero, bh, s, d, group, bits, y),
           "dequantize_keys")
    return y


def dequantize_values(codes, scale, zero, group: int, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    zero = np.ascontiguousarray(zero, dtype=np.float32)
    bh, s, dw = codes.shape
    d = dw * codes_per_word(bits)
    y = np.zeros((bh, s, d), np.uint16)
    _check(lib().kivi_oracle_dequantize_values(codes, scale, zero, bh, s, d, group, bits, y),
           "dequantize_values")
    return y


def key_group(x_bh: np.ndarray, g: int, c: int, group: int, bits: int):
    """One key group of a [s, d] slice: (words u32 [G/W], scale, zero)."""
    x_bh = np.ascontiguousarray(x_bh, dtype=np.uint16)
    s, d = x_bh.shape
    words = np.zeros(group // codes_per_word(bits), np.uint32)
    sc, ze = C.c_float(), C.c_float()
    _check(lib().kivi_oracle_key_group(x_bh, s, d, g, c, group, bits, words,
                                       C.byref(sc), C.byref(ze)), "key_group")
    return words, np.float32(sc.value), np.float32(ze.value)


def value_row(x_row: np.ndarray, group: int, bits: int):
    """One value row [d]: (words u32 [d/W], scale f32 [d/G], zero f32 [d/G])."""
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16).reshape(-1)
    d = x_row.size
    words = np.zeros(d // codes_per_word(bits), np.uint32)
    scale = np.zeros(d // group, np.float32)
    zero = np.zeros(d // group, np.float32)
    _check(lib().kivi_oracle_value_row(x_row, d, group, bits, words, scale, zero), "value_row")
    return words, scale, zero


def flush_size(n_res: int, residual: int, group: int) -> int:
    return int(lib().kivi_oracle_flush_size(n_res, residual, group))


class Store:
    """Host-side quantized store of one layer (oracle layout, capacity ``cap`` tokens)."""

    def __init__(self, bh: int, d: int, cap: int, group: int, bits: int):
        w = codes_per_word(bits)
        self.bh, self.d, self.cap, self.group, self.bits = bh, d, cap, group, bits
        self.k_codes = np.zeros((bh, cap // w, d), np.uint32)
        self.k_scale = np.zeros((bh, cap // group, d), np.float32)
        self.k_zero = np.zeros((bh, cap // group, d), np.float32)
        self.v_codes = np.zeros((bh, cap, d // w), np.uint32)
        self.v_scale = np.zeros((bh, cap, d // group), np.float32)
        self.v_zero = np.zeros((bh, cap, d // group), np.float32)


def append(k_res: np.ndarray, v_res: np.ndarray, res_head: int, n_res: int,
           k_new: np.ndarray, v_new: np.ndarray) -> int:
    """Writes new tokens k_new, v_new [bh, n, d] (fp16 bits) behind the
    residual of the rings k_res, v_res [bh, r_cap, d] (in place); returns the
    new residual count."""
    bh, r_cap, d = k_res.shape
    assert k_res.flags.c_contiguous and v_res.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    cnt = C.c_int64(n_res)
    _check(lib().kivi_oracle_append(k_res, v_res, bh, d, r_cap, res_head, C.byref(cnt), k_new,
                                    v_new, k_new.shape[1]), "append")
    return int(cnt.value)


def flush(k_res: np.ndarray, v_res: np.ndarray, store: Store, residual: int,
          s_q: int, res_head: int, n_res: int):
    """Flush one layer's residual ring into ``store``.

    Returns ``(n_flushed, s_q, res_head, n_res)`` after the flush.
    """
    k_res = np.ascontiguousarray(k_res, dtype=np.uint16)
    v_res = np.ascontiguousarray(v_res, dtype=np.uint16)
    bh, r_cap, d = k_res.shape
    a, b, c = C.c_int64(s_q), C.c_int64(res_head), C.c_int64(n_res)
    n = lib().kivi_oracle_flush(k_res, v_res, bh, d, r_cap, store.cap, store.group,
                                store.bits, residual, store.k_codes, store.k_scale,
                                store.k_zero, store.v_codes, store.v_scale, store.v_zero,
                                C.byref(a), C.byref(b), C.byref(c))
    if n < 0:
        raise ValueError(f"oracle flush rejected its arguments (rc={n})")
    return int(n), a.value, b.value, c.value


# ---------------------------------------------------------------------------
# decode attention over the reconstructed cache
# ---------------------------------------------------------------------------

def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Attention of the query rows q [r, d] (fp16 bits) over the tokens of one
    KV head, keys k and values v [n, d] (fp16 bits), in binary64 -> [r, d]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    r, d = q.shape
    n = k.shape[0]
    if k.shape != (n, d) or v.shape != (n, d):
        raise ValueError("k and v must be [n, d] with the query's d")
    out = np.zeros((r, d), np.float64)
    _check(lib().kivi_oracle_attention(q, r, k, v, n, d, float(scale), out), "attention")
    return out


def decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Grouped-query decode attention: q [batch, h_q, d]; k, v [batch*h_kv, n, d]
    (fp16 bits).  Query head h of sequence b attends KV head b*h_kv + h // (h_q/h_kv)
    (consecutive query heads share a KV head).  Returns [batch, h_q, d] binary64."""
    batch, h_q, d = q.shape
    bh = k.shape[0]
    h_kv = bh // batch
    if h_kv * batch != bh or h_q % h_kv:
        raise ValueError("inconsistent head counts")
    r = h_q // h_kv
    out = np.zeros((batch, h_q, d), np.float64)
    for b in range(batch):
        for j in range(h_kv):
            out[b, j * r:(j + 1) * r] = attention(q[b, j * r:(j + 1) * r], k[b * h_kv + j],
                                                  v[b * h_kv + j], scale)
    return out


def cache_kv(store: Store, s_q: int, k_ring: np.ndarray, v_ring: np.ndarray, res_head: int,
             n_res: int):
    """The fp16 keys and values a cache holds, in token order: the first s_q
    store tokens dequantized, then the n_res residual tokens of the rings
    [bh, r_cap, d] read from ring row res_head on.  Returns (k, v), each
    [bh, s_q + n_res, d] fp16 bits."""
    w = codes_per_word(store.bits)
    g = store.group
    parts_k, parts_v = [], []
    if s_q:
        parts_k.append(dequantize_keys(store.k_codes[:, :s_q // w], store.k_scale[:, :s_q // g],
                                       store.k_zero[:, :s_q // g], s_q, g, store.bits))
        parts_v.append(dequantize_values(store.v_codes[:, :s_q], store.v_scale[:, :s_q],
                                         store.v_zero[:, :s_q], g, store.bits))
    if n_res:
        rows = (res_head + np.arange(n_res)) % k_ring.shape[1]
        parts_k.append(k_ring[:, rows])
        parts_v.append(v_ring[:, rows])
    return (np.ascontiguousarray(np.concatenate(parts_k, axis=1)),
            np.ascontiguousarray(np.concatenate(parts_v, axis=1)))


# ---------------------------------------------------------------------------
# KIVI-Sink
# ---------------------------------------------------------------------------

def sink_scores(k: np.ndarray, heads: int) -> np.ndarray:
    """Key-norm scores of k [batch*heads, n, d] (fp16 bits) -> float32 [batch, n]:
    the mean over the KV heads of each token's key L2 norm."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    bh, n, d = k.shape
    batch = bh // heads
    out = np.zeros((batch, n), np.float32)
    _check(lib().kivi_oracle_sink_scores(k, batch, heads, n, d, n * d, out), "sink_scores")
    return out


class SinkState:
    """Running top-k positions of every sequence and the sink store of one layer."""

    def __init__(self, batch: int, heads: int, d: int, k_top: int, sink_cap: int):
        self.batch, self.heads, self.d, self.k_top, self.sink_cap = batch, heads, d, k_top, sink_cap
        self.top_pos = np.zeros((batch, max(k_top, 1)), np.int64)
        self.top_score = np.zeros((batch, max(k_top, 1)), np.float32)
        self.top_count = np.zeros(batch, np.int64)
        self.sink_pos = np.zeros((batch, max(sink_cap, 1)), np.int64)
        self.sink_count = np.zeros(batch, np.int64)
        self.sink_k = np.zeros((batch * heads, max(sink_cap, 1), d), np.uint16)
        self.sink_v = np.zeros((batch * heads, max(sink_cap, 1), d), np.uint16)

    def update(self, scores: np.ndarray, p0: int) -> None:
        """Merge the scores [batch, n] of positions p0 .. p0+n-1 into the top-k."""
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        for b in range(self.batch):
            pos = np.ascontiguousarray(self.top_pos[b])
            sc = np.ascontiguousarray(self.top_score[b])
            cnt = C.c_int64(int(self.top_count[b]))
            _check(lib().kivi_oracle_sink_topk(self.k_top, pos, sc, C.byref(cnt),
                                               np.ascontiguousarray(scores[b]), p0,
                                               scores.shape[1]), "sink_topk")
            self.top_pos[b], self.top_score[b], self.top_count[b] = pos, sc, cnt.value


def flush_sink(k_res: np.ndarray, v_res: np.ndarray, store: "Store", residual: int, s_q: int,
               res_head: int, n_res: int, state: SinkState):
    """Flush with sink protection; returns ``(n_flushed, s_q, res_head, n_res)``."""
    k_res = np.ascontiguousarray(k_res, dtype=np.uint16)
    v_res = np.ascontiguousarray(v_res, dtype=np.uint16)
    bh, r_cap, d = k_res.shape
    a, b, c = C.c_int64(s_q), C.c_int64(res_head), C.c_int64(n_res)
    n = lib().kivi_oracle_flush_sink(
        k_res, v_res, state.batch, state.heads, d, r_cap, store.cap, store.group, store.bits,
        residual, store.k_codes, store.k_scale, store.k_zero, store.v_codes, store.v_scale,
        store.v_zero, C.byref(a), C.byref(b), C.byref(c), state.top_pos.shape[1],
        state.top_pos, state.top_count, state.sink_pos.shape[1], state.sink_pos,
        state.sink_count, state.sink_k, state.sink_v)
    if n < 0:
        raise ValueError(f"oracle sink flush rejected its arguments (rc={n})")
    return int(n), a.value, b.value, c.value


def sink_restore(k: np.ndarray, v: np.ndarray, state: SinkState) -> None:
    """Put the sink rows back into dequantized k, v [bh, s, d] (in place)."""
    bh, s, d = k.shape
    _check(lib().kivi_oracle_sink_restore(k, v, state.batch, state.heads, s, d,
                                          state.sink_pos.shape[1], state.sink_pos,
                                          state.sink_count, state.sink_k, state.sink_v),
           "sink_restore")
