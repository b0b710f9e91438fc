"""Python binding of ``libkivi`` -- the GB300 KIVI KV-cache codec.

Argument marshalling only: every step of quantization, dequantization and
flush runs in the library's CUDA kernels (``csrc/``); PyTorch supplies device
memory and streams.  The functions carry the names of the C entry points
declared in ``include/kivi.h`` and take ``torch`` CUDA tensors:

    fp16 tensors       torch.float16, shape [bh, s, d], last two dims contiguous
    code words         torch.int32 (bit patterns of the uint32 words)
    scales and zeros   torch.float32

If the shared library is missing it is built from ``csrc/`` with nvcc; if
that is impossible the import of :func:`lib` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import List, Optional, Sequence, Tuple

from . import _build

__all__ = [
    "KiviError", "lib", "library_path", "debug_bounds", "kivi_quantize_keys", "kivi_quantize_values",
    "kivi_dequantize_keys", "kivi_dequantize_values", "kivi_flush", "kivi_flush_size",
    "kivi_append", "kivi_append_flush",
    "kivi_dequantize_cache", "kivi_key_code_words", "kivi_value_code_words",
    "kivi_fakequant_keys", "kivi_fakequant_values", "kivi_flush_fakequant",
    "kivi_decode_attention", "kivi_decode_attention_splits", "kivi_decode_attention_workspace",
    "kivi_decode_attention_noalloc", "kivi_decode_attention_sinks", "kivi_device_fault",
    "kivi_selftest_wait_timeout",
    "kivi_sink_update", "kivi_flush_sink",
    "kivi_sink_restore", "kivi_sink_layer", "kivi_sink_cfg", "KiviSinks",
    "KiviCache", "kivi_layer", "kivi_cache", "STATUS",
    "KIVI_MAX_LAYERS", "event_handles",
]

KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN, KIVI_ERR_CAPACITY, KIVI_ERR_CUDA = range(5)
STATUS = {0: "KIVI_OK", 1: "KIVI_ERR_INVAL", 2: "KIVI_ERR_ALIGN", 3: "KIVI_ERR_CAPACITY",
          4: "KIVI_ERR_CUDA"}
KIVI_MAX_LAYERS = 128


class KiviError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if _lib is not None:
            msg += f" ({_lib.kivi_status_string(status).decode()})"
            if status == KIVI_ERR_CUDA:
                msg += f", cudaError {_lib.kivi_last_cuda_error()}"
        super().__init__(msg)


class kivi_layer(C.Structure):
    _fields_ = [("k_res", C.c_void_p), ("v_res", C.c_void_p), ("k_codes", C.c_void_p),
                ("k_scale", C.c_void_p), ("k_zero", C.c_void_p), ("v_codes", C.c_void_p),
                ("v_scale", C.c_void_p), ("v_zero", C.c_void_p)]


class kivi_cache(C.Structure):
    _fields_ = [("bh", C.c_int64), ("d", C.c_int64), ("r_cap", C.c_int64), ("cap", C.c_int64),
                ("group", C.c_int32), ("bits", C.c_int32), ("residual", C.c_int32),
                ("reserved", C.c_int32), ("s_q", C.c_int64), ("res_head", C.c_int64),
                ("n_res", C.c_int64)]


class kivi_sink_layer(C.Structure):
    _fields_ = [("top_pos", C.c_void_p), ("top_score", C.c_void_p), ("top_count", C.c_void_p),
                ("sink_pos", C.c_void_p), ("sink_count", C.c_void_p), ("sink_k", C.c_void_p),
                ("sink_v", C.c_void_p), ("mask", C.c_void_p), ("scores", C.c_void_p)]


class kivi_sink_cfg(C.Structure):
    _fields_ = [("batch", C.c_int64), ("k_top", C.c_int32), ("sink_cap", C.c_int32),
                ("reserved", C.c_int32), ("reserved2", C.c_int32)]


_lock = threading.Lock()
_lib = None

_i64, _int, _vp = C.c_int64, C.c_int, C.c_void_p


def debug_bounds() -> bool:
    """True when ``KIVI_DEBUG_BOUNDS=1``: the index-checking build is loaded."""
    return os.environ.get("KIVI_DEBUG_BOUNDS") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_bounds() else _build.LIB_PATH


def lib():
    """The loaded ``libkivi.so`` (built from source first if missing; with
    ``KIVI_DEBUG_BOUNDS=1`` the index-checking ``libkivi_debug.so``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build(debug_bounds=debug_bounds())
            L = C.CDLL(path)
            q_args = [_vp, _i64, _i64, _i64, _i64, _int, _int, _vp, _i64, _vp, _vp, _i64, _vp]
            dq_args = [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _vp, _i64, _vp]
            fq_args = [_vp, _i64, _i64, _i64, _i64, _int, _int, _vp, _i64, _vp, _i64, _vp, _vp,
                       _i64, _vp]
            for name, args in (("kivi_quantize_keys", q_args), ("kivi_quantize_values", q_args),
                               ("kivi_fakequant_keys", fq_args),
                               ("kivi_fakequant_values", fq_args),
                               ("kivi_dequantize_keys", dq_args),
                               ("kivi_dequantize_values", dq_args)):
                f = getattr(L, name)
                f.argtypes = args
                f.restype = _int
            L.kivi_flush.argtypes = [C.POINTER(kivi_layer), _int, C.POINTER(kivi_cache),
                                     C.POINTER(_i64), _vp]
            L.kivi_flush.restype = _int
            L.kivi_append.argtypes = [C.POINTER(kivi_layer), _int, C.POINTER(kivi_cache),
                                      C.POINTER(_vp), C.POINTER(_vp), _i64, _i64, _vp]
            L.kivi_append.restype = _int
            L.kivi_append_flush.argtypes = [C.POINTER(kivi_layer), _int, C.POINTER(kivi_cache),
                                            C.POINTER(_vp), C.POINTER(_vp), _i64, _i64,
                                            C.POINTER(_i64), _vp, C.POINTER(_vp)]
            L.kivi_append_flush.restype = _int
            L.kivi_dequantize_cache.argtypes = [C.POINTER(kivi_layer), _int,
                                                C.POINTER(kivi_cache), C.POINTER(_vp),
                                                C.POINTER(_vp), _vp]
            L.kivi_dequantize_cache.restype = _int
            L.kivi_flush_timed.argtypes = [C.POINTER(kivi_layer), _int, C.POINTER(kivi_cache),
                                           C.POINTER(_i64), _vp, C.POINTER(_vp)]
            L.kivi_flush_timed.restype = _int
            L.kivi_dequantize_cache_timed.argtypes = [C.POINTER(kivi_layer), _int,
                                                      C.POINTER(kivi_cache), C.POINTER(_vp),
                                                      C.POINTER(_vp), _vp, C.POINTER(_vp)]
            L.kivi_dequantize_cache_timed.restype = _int
            L.kivi_flush_fakequant.argtypes = [C.POINTER(kivi_layer), _int, C.POINTER(kivi_cache),
                                               C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_i64),
                                               _vp, C.POINTER(_vp)]
            L.kivi_flush_fakequant.restype = _int
            L.kivi_decode_attention.argtypes = [C.POINTER(kivi_layer), _int,
                                                C.POINTER(kivi_cache), _i64, C.c_int32,
                                                C.c_float, C.POINTER(_vp), C.POINTER(_vp),
                                                C.c_int32, _vp, _i64, _vp]
            L.kivi_decode_attention.restype = _int
            L.kivi_decode_attention_sinks.argtypes = [C.POINTER(kivi_layer),
                                                      C.POINTER(kivi_sink_layer), _int,
                                                      C.POINTER(kivi_cache),
                                                      C.POINTER(kivi_sink_cfg), _i64, C.c_int32,
                                                      C.c_float, C.POINTER(_vp), C.POINTER(_vp),
                                                      C.c_int32, _vp, _i64, _vp]
            L.kivi_decode_attention_sinks.restype = _int
            L.kivi_decode_attention_splits.argtypes = [C.POINTER(kivi_cache), _int, _i64]
            L.kivi_decode_attention_splits.restype = C.c_int32
            L.kivi_decode_attention_workspace.argtypes = [C.POINTER(kivi_cache), _int, _i64,
                                                          C.c_int32, C.c_int32]
            L.kivi_decode_attention_workspace.restype = _i64
            L.kivi_decode_attention_noalloc.argtypes = [C.POINTER(kivi_layer), _int,
                                                        C.POINTER(kivi_cache), _i64, C.c_int32,
                                                        C.c_float, C.POINTER(_vp),
                                                        C.POINTER(_vp), C.c_int32, _vp]
            L.kivi_decode_attention_noalloc.restype = _int
            L.kivi_sink_update.argtypes = [C.POINTER(kivi_layer), C.POINTER(kivi_sink_layer),
                                           _int, C.POINTER(kivi_cache), C.POINTER(kivi_sink_cfg),
                                           _i64, _i64, _vp]
            L.kivi_sink_update.restype = _int
            L.kivi_flush_sink.argtypes = [C.POINTER(kivi_layer), C.POINTER(kivi_sink_layer), _int,
                                          C.POINTER(kivi_cache), C.POINTER(kivi_sink_cfg),
                                          C.POINTER(_i64), _vp]
            L.kivi_flush_sink.restype = _int
            L.kivi_sink_restore.argtypes = [C.POINTER(kivi_sink_layer), _int, C.POINTER(kivi_cache),
                                            C.POINTER(kivi_sink_cfg), C.POINTER(_vp),
                                            C.POINTER(_vp), _vp]
            L.kivi_sink_restore.restype = _int
            L.kivi_device_fault.argtypes = [C.POINTER(C.c_uint32)]
            L.kivi_device_fault.restype = _int
            L.kivi_selftest_wait_timeout.argtypes = [C.c_uint32, _vp]
            L.kivi_selftest_wait_timeout.restype = _int
            L.kivi_flush_size.argtypes = [_i64, _int, _int]
            L.kivi_flush_size.restype = _i64
            L.kivi_key_code_words.argtypes = [_i64, _i64, _int, _int]
            L.kivi_key_code_words.restype = _i64
            L.kivi_value_code_words.argtypes = [_i64, _i64, _int, _int]
            L.kivi_value_code_words.restype = _i64
            L.kivi_status_string.argtypes = [_int]
            L.kivi_status_string.restype = C.c_char_p
            L.kivi_last_cuda_error.argtypes = []
            L.kivi_last_cuda_error.restype = _int
            L.kivi_abi_version.argtypes = []
            L.kivi_abi_version.restype = _int
            _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != KIVI_OK:
        raise KiviError(status, where)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream))


def _fp16_3d(x, what: str):
    import torch
    if x.dtype != torch.float16 or x.dim() != 3 or not x.is_cuda:
        raise ValueError(f"{what}: expected a CUDA float16 tensor [bh, s, d]")
    if x.shape[1] > 0 and x.shape[2] > 0 and (x.stride(2) != 1 or x.stride(1) != x.shape[2]):
        raise ValueError(f"{what}: the last two dimensions must be contiguous")
    return x


def _bh_stride(t) -> int:
    return int(t.stride(0)) if t.shape[0] > 1 else int(t[0].numel()) if t.numel() else 0


def codes_per_word(bits: int) -> int:
    return 32 // bits


def kivi_flush_size(n_res: int, residual: int, group: int) -> int:
    return int(lib().kivi_flush_size(n_res, residual, group))


def kivi_key_code_words(s: int, d: int, group: int, bits: int) -> int:
    return int(lib().kivi_key_code_words(s, d, group, bits))


def kivi_value_code_words(s: int, d: int, group: int, bits: int) -> int:
    return int(lib().kivi_value_code_words(s, d, group, bits))


# ---------------------------------------------------------------------------
# full-tensor calls
# ---------------------------------------------------------------------------

def kivi_quantize_keys(x, group: int, bits: int, codes=None, scale=None, zero=None,
                       stream=None) -> Tuple:
    """Per-channel key quantization of x [bh, s, d] -> (codes [bh, ng*G/W, d] int32,
    scale [bh, ng, d] f32, zero [bh, ng, d] f32)."""
    import torch
    x = _fp16_3d(x, "kivi_quantize_keys")
    bh, s, d = x.shape
    ng = -(-s // group)
    if codes is None:
        codes = torch.empty((bh, ng * group // codes_per_word(bits), d), dtype=torch.int32,
                            device=x.device)
    if scale is None:
        scale = torch.empty((bh, ng, d), dtype=torch.float32, device=x.device)
    if zero is None:
        zero = torch.empty((bh, ng, d), dtype=torch.float32, device=x.device)
    _check(lib().kivi_quantize_keys(x.data_ptr(), bh, s, d, _bh_stride(x), group, bits,
                                    codes.data_ptr(), _bh_stride(codes), scale.data_ptr(),
                                    zero.data_ptr(), _bh_stride(scale), _stream_handle(stream)),
           "kivi_quantize_keys")
    return codes, scale, zero


def kivi_quantize_values(x, group: int, bits: int, codes=None, scale=None, zero=None,
                         stream=None) -> Tuple:
    """Per-token value quantization of x [bh, s, d] -> (codes [bh, s, d/W] int32,
    scale [bh, s, d/G] f32, zero [bh, s, d/G] f32)."""
    import torch
    x = _fp16_3d(x, "kivi_quantize_values")
    bh, s, d = x.shape
    if codes is None:
        codes = torch.empty((bh, s, d // codes_per_word(bits)), dtype=torch.int32,
                            device=x.device)
    if scale is None:
        scale = torch.empty((bh, s, max(1, d // group)), dtype=torch.float32, device=x.device)
    if zero is None:
        zero = torch.empty((bh, s, max(1, d // group)), dtype=torch.float32, device=x.device)
    _check(lib().kivi_quantize_values(x.data_ptr(), bh, s, d, _bh_stride(x), group, bits,
                                      codes.data_ptr(), _bh_stride(codes), scale.data_ptr(),
                                      zero.data_ptr(), _bh_stride(scale), _stream_handle(stream)),
           "kivi_quantize_values")
    return codes, scale, zero


def kivi_dequantize_keys(codes, scale, zero, s: int, group: int, bits: int, y=None,
                         stream=None):
    """Key reconstruction [bh, s, d] fp16 from the key code layout."""
    import torch
    bh, _, d = codes.shape
    if y is None:
        y = torch.empty((bh, s, d), dtype=torch.float16, device=codes.device)
    _check(lib().kivi_dequantize_keys(codes.data_ptr(), _bh_stride(codes), scale.data_ptr(),
                                      zero.data_ptr(), _bh_stride(scale), bh, s, d, group, bits,
                                      y.data_ptr(), _bh_stride(y), _stream_handle(stream)),
           "kivi_dequantize_keys")
    return y


def kivi_dequantize_values(codes, scale, zero, group: int, bits: int, s: Optional[int] = None,
                           y=None, stream=None):
    """Value reconstruction [bh, s, d] fp16 from the value code layout."""
    import torch
    bh, s_codes, dw = codes.shape
    s = s_codes if s is None else s
    d = dw * codes_per_word(bits)
    if y is None:
        y = torch.empty((bh, s, d), dtype=torch.float16, device=codes.device)
    _check(lib().kivi_dequantize_values(codes.data_ptr(), _bh_stride(codes), scale.data_ptr(),
                                        zero.data_ptr(), _bh_stride(scale), bh, s, d, group,
                                        bits, y.data_ptr(), _bh_stride(y),
                                        _stream_handle(stream)),
           "kivi_dequantize_values")
    return y


def _fakequant(name: str, x, group: int, bits: int, y, store: bool, codes, scale, zero,
               stream, shapes):
    import torch
    x = _fp16_3d(x, name)
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    y = _fp16_3d(y, name + " (y)")
    if store:
        cs, ss = shapes
        codes = torch.empty(cs, dtype=torch.int32, device=x.device) if codes is None else codes
        scale = torch.empty(ss, dtype=torch.float32, device=x.device) if scale is None else scale
        zero = torch.empty(ss, dtype=torch.float32, device=x.device) if zero is None else zero
        cp, cst, sp, zp, sst = (codes.data_ptr(), _bh_stride(codes), scale.data_ptr(),
                                zero.data_ptr(), _bh_stride(scale))
    else:
        codes = scale = zero = None
        cp, cst, sp, zp, sst = None, 0, None, None, 0
    bh, s, d = x.shape
    _check(getattr(lib(), name)(x.data_ptr(), bh, s, d, _bh_stride(x), group, bits, y.data_ptr(),
                                _bh_stride(y), cp, cst, sp, zp, sst, _stream_handle(stream)), name)
    return y, codes, scale, zero


def kivi_fakequant_keys(x, group: int, bits: int, y=None, store: bool = True, codes=None,
                        scale=None, zero=None, stream=None) -> Tuple:
    """Fused per-channel key quantize + dequantize of x [bh, s, d] in one pass ->
    (y [bh, s, d] fp16, codes, scale, zero); with ``store=False`` only y is
    written and the last three are None."""
    bh, s, d = x.shape
    ng = -(-s // group)
    return _fakequant("kivi_fakequant_keys", x, group, bits, y, store, codes, scale, zero, stream,
                      ((bh, ng * group // codes_per_word(bits), d), (bh, ng, d)))


def kivi_fakequant_values(x, group: int, bits: int, y=None, store: bool = True, codes=None,
                          scale=None, zero=None, stream=None) -> Tuple:
    """Fused per-token value quantize + dequantize of x [bh, s, d] in one pass ->
    (y [bh, s, d] fp16, codes, scale, zero); with ``store=False`` only y."""
    bh, s, d = x.shape
    return _fakequant("kivi_fakequant_values", x, group, bits, y, store, codes, scale, zero,
                      stream, ((bh, s, d // codes_per_word(bits)), (bh, s, max(1, d // group))))


# ---------------------------------------------------------------------------
# cache: residual ring + quantized store, flush, batched dequantization
# ---------------------------------------------------------------------------

def event_handles(events) -> "C.Array":
    """ctypes array of three cudaEvent_t handles from torch.cuda.Event objects
    (each must have been recorded once so that the CUDA event exists)."""
    return (C.c_void_p * 3)(*[e.cuda_event if e is not None else None for e in events])


def kivi_flush(layers, n_layers: int, cache: kivi_cache, stream=None, events=None) -> int:
    """Raw C call: ``layers`` a ctypes array of kivi_layer, ``cache`` a kivi_cache
    (updated in place).  ``events``: optional (ctypes array of) three event
    handles recorded around the two launches.  Returns the tokens flushed."""
    n = C.c_int64(0)
    if events is None:
        st = lib().kivi_flush(layers, n_layers, C.byref(cache), C.byref(n),
                              _stream_handle(stream))
    else:
        if not isinstance(events, C.Array):
            events = event_handles(events)
        st = lib().kivi_flush_timed(layers, n_layers, C.byref(cache), C.byref(n),
                                    _stream_handle(stream), events)
    _check(st, "kivi_flush")
    return int(n.value)


def _ptr_array(ts, n: int):
    return ts if isinstance(ts, C.Array) else (C.c_void_p * n)(*[t.data_ptr() for t in ts])


def kivi_append_flush(layers, n_layers: int, cache: kivi_cache, k_new, v_new, n: int,
                      new_bh_stride: int, stream=None, events=None) -> int:
    """Raw C call: append + flush in one call (``k_new``/``v_new`` prepared
    ctypes pointer arrays or per-layer tensors, ``new_bh_stride`` in
    elements); ``events`` None or four cudaEvent handles / torch events.
    Returns the tokens flushed."""
    out = C.c_int64(0)
    if events is not None and not isinstance(events, C.Array):
        events = (C.c_void_p * 4)(*[e.cuda_event if e is not None else None for e in events])
    _check(lib().kivi_append_flush(layers, n_layers, C.byref(cache), _ptr_array(k_new, n_layers),
                                   _ptr_array(v_new, n_layers), new_bh_stride, n, C.byref(out),
                                   _stream_handle(stream), events), "kivi_append_flush")
    return int(out.value)


def kivi_append(layers, n_layers: int, cache: kivi_cache, k_new, v_new, n: int,
                new_bh_stride: Optional[int] = None, stream=None) -> None:
    """Raw C call: new tokens of every layer into the residual rings behind the
    residual (``cache.n_res`` advances by n).  ``k_new``/``v_new``: sequences
    of fp16 [bh, n, d] tensors (last two dims contiguous) or prepared ctypes
    pointer arrays (then ``new_bh_stride``, in elements, is required)."""
    if new_bh_stride is None:
        t = k_new[0]
        for x in list(k_new) + list(v_new):
            _fp16_3d(x, "kivi_append")
            if _bh_stride(x) != _bh_stride(t):
                raise ValueError("kivi_append: every new-token tensor needs the same bh stride")
        new_bh_stride = _bh_stride(t)
    _check(lib().kivi_append(layers, n_layers, C.byref(cache), _ptr_array(k_new, n_layers),
                             _ptr_array(v_new, n_layers), new_bh_stride, n,
                             _stream_handle(stream)), "kivi_append")


def kivi_flush_fakequant(layers, n_layers: int, cache: kivi_cache, k_hat, v_hat, stream=None,
                         events=None) -> int:
    """Raw C call of the fused fake-quant flush: as :func:`kivi_flush`, and the
    fp16 reconstruction of the flushed tokens goes to rows s_q .. of
    ``k_hat[l]``/``v_hat[l]`` (fp16 [bh, cap, d] tensors or ctypes pointer
    arrays).  Returns the tokens flushed."""
    n = C.c_int64(0)
    if events is not None and not isinstance(events, C.Array):
        events = event_handles(events)
    st = lib().kivi_flush_fakequant(layers, n_layers, C.byref(cache), _ptr_array(k_hat, n_layers),
                                    _ptr_array(v_hat, n_layers), C.byref(n),
                                    _stream_handle(stream), events)
    _check(st, "kivi_flush_fakequant")
    return int(n.value)


def kivi_dequantize_cache(layers, n_layers: int, cache: kivi_cache, k_out, v_out,
                          stream=None, events=None) -> None:
    """``k_out``/``v_out``: sequences of fp16 tensors, or prepared ctypes pointer arrays."""
    kp = _ptr_array(k_out, n_layers)
    vp = _ptr_array(v_out, n_layers)
    if events is None:
        st = lib().kivi_dequantize_cache(layers, n_layers, C.byref(cache), kp, vp,
                                         _stream_handle(stream))
    else:
        if not isinstance(events, C.Array):
            events = event_handles(events)
        st = lib().kivi_dequantize_cache_timed(layers, n_layers, C.byref(cache), kp, vp,
                                               _stream_handle(stream), events)
    _check(st, "kivi_dequantize_cache")


def kivi_decode_attention_splits(cache: kivi_cache, n_layers: int, batch: int) -> int:
    return int(lib().kivi_decode_attention_splits(C.byref(cache), n_layers, batch))


def kivi_decode_attention_workspace(cache: kivi_cache, n_layers: int, batch: int, h_q: int,
                                    n_split: int) -> int:
    return int(lib().kivi_decode_attention_workspace(C.byref(cache), n_layers, batch, h_q,
                                                     n_split))


def kivi_decode_attention(layers, n_layers: int, cache: kivi_cache, batch: int, h_q: int,
                          sm_scale: float, q, out, n_split: int = 1, workspace=None,
                          stream=None) -> None:
    """Raw C call: ``q``/``out`` sequences of per-layer tensors (fp16 / fp32
    [batch, h_q, d]) or prepared ctypes pointer arrays; ``workspace`` a float32
    tensor of at least :func:`kivi_decode_attention_workspace` elements when
    ``n_split > 1``."""
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _check(lib().kivi_decode_attention(layers, n_layers, C.byref(cache), batch, h_q,
                                       float(sm_scale), _ptr_array(q, n_layers),
                                       _ptr_array(out, n_layers), n_split, wp, wn,
                                       _stream_handle(stream)),
           "kivi_decode_attention")


def kivi_decode_attention_sinks(layers, sinks, n_layers: int, cache: kivi_cache,
                                cfg: "kivi_sink_cfg", batch: int, h_q: int, sm_scale: float, q,
                                out, n_split: int = 1, workspace=None, stream=None) -> None:
    """As :func:`kivi_decode_attention`, over a sink-protected cache: the stored
    sinks' exact fp16 rows replace their store slots."""
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _check(lib().kivi_decode_attention_sinks(layers, sinks, n_layers, C.byref(cache),
                                             C.byref(cfg), batch, h_q, float(sm_scale),
                                             _ptr_array(q, n_layers), _ptr_array(out, n_layers),
                                             n_split, wp, wn, _stream_handle(stream)),
           "kivi_decode_attention_sinks")


def kivi_decode_attention_noalloc(layers, n_layers: int, cache: kivi_cache, batch: int,
                                  h_q: int, sm_scale: float, q, out, n_split: int = 1,
                                  stream=None) -> None:
    """As :func:`kivi_decode_attention`, the split workspace being the library's
    fixed device array (no workspace argument, nothing allocated; calls that
    overlap on the device race)."""
    _check(lib().kivi_decode_attention_noalloc(layers, n_layers, C.byref(cache), batch, h_q,
                                               float(sm_scale), _ptr_array(q, n_layers),
                                               _ptr_array(out, n_layers), n_split,
                                               _stream_handle(stream)),
           "kivi_decode_attention_noalloc")


def kivi_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Raw C call: one warp's bounded wait on a phase nothing completes; bit 2
    of the device fault word is set once it gives up (asynchronous)."""
    _check(lib().kivi_selftest_wait_timeout(limit_us, _stream_handle(stream)),
           "kivi_selftest_wait_timeout")


def kivi_device_fault() -> int:
    """Reads and clears the device fault word (nonzero: a pipeline wait gave up)."""
    v = C.c_uint32(0)
    _check(lib().kivi_device_fault(C.byref(v)), "kivi_device_fault")
    return int(v.value)


class KiviCache:
    """Device buffers and state of an ``n_layers`` KIVI cache (all torch-allocated).

    Per layer: fp16 residual rings ``k_res``/``v_res`` [bh, r_cap, d] and the
    quantized store (key codes [bh, cap/W, d], key scale/zero [bh, cap/G, d],
    value codes [bh, cap, d/W], value scale/zero [bh, cap, d/G]).  With
    ``recon=True`` also fp16 reconstructions ``k_hat``/``v_hat`` [bh, cap, d]
    that :meth:`flush_fakequant` fills; ``store=False`` (only with recon)
    leaves the quantized store out: the cache then holds the reconstruction
    alone.
    """

    def __init__(self, n_layers: int, bh: int, d: int, r_cap: int, cap: int, group: int = 32,
                 bits: int = 2, residual: int = 32, device="cuda", recon: bool = False,
                 store: bool = True):
        import torch
        if not (1 <= n_layers <= KIVI_MAX_LAYERS):
            raise ValueError("n_layers out of range")
        w = codes_per_word(bits)
        self.n_layers, self.group, self.bits = n_layers, group, bits
        dev = torch.device(device)
        # one contiguous allocation per buffer kind, one view per layer
        if not store and not recon:
            raise ValueError("a cache without a store needs recon=True")
        mk = lambda shape, dt: torch.zeros((n_layers,) + shape, dtype=dt, device=dev)  # noqa
        self.k_res_all = mk((bh, r_cap, d), torch.float16)
        self.v_res_all = mk((bh, r_cap, d), torch.float16)
        self.k_res = list(self.k_res_all.unbind(0))
        self.v_res = list(self.v_res_all.unbind(0))
        names = ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero")
        if store:
            shapes = ((bh, cap // w, d), (bh, cap // group, d), (bh, cap // group, d),
                      (bh, cap, d // w), (bh, cap, d // group), (bh, cap, d // group))
            dts = (torch.int32, torch.float32, torch.float32) * 2
            for name, shape, dt in zip(names, shapes, dts):
                setattr(self, name + "_all", mk(shape, dt))
                setattr(self, name, list(getattr(self, name + "_all").unbind(0)))
        else:
            for name in names:
                setattr(self, name + "_all", None)
                setattr(self, name, [None] * n_layers)
        self.recon = recon
        self.k_hat_all = mk((bh, cap, d), torch.float16) if recon else None
        self.v_hat_all = mk((bh, cap, d), torch.float16) if recon else None
        self.k_hat = list(self.k_hat_all.unbind(0)) if recon else None
        self.v_hat = list(self.v_hat_all.unbind(0)) if recon else None
        ptr = lambda t: t.data_ptr() if t is not None else None  # noqa
        self.layers = (kivi_layer * n_layers)(*[
            kivi_layer(self.k_res[i].data_ptr(), self.v_res[i].data_ptr(),
                       *[ptr(getattr(self, name)[i]) for name in names])
            for i in range(n_layers)])
        if recon:
            self._k_hat_ptrs = _ptr_array(self.k_hat, n_layers)
            self._v_hat_ptrs = _ptr_array(self.v_hat, n_layers)
        self.state = kivi_cache(bh, d, r_cap, cap, group, bits, residual, 0, 0, 0, 0)

    # state ------------------------------------------------------------------
    @property
    def s_q(self) -> int:
        return int(self.state.s_q)

    @property
    def n_res(self) -> int:
        return int(self.state.n_res)

    @property
    def res_head(self) -> int:
        return int(self.state.res_head)

    def reset(self, s_q: int = 0, res_head: int = 0, n_res: int = 0) -> None:
        self.state.s_q, self.state.res_head, self.state.n_res = s_q, res_head, n_res

    def append(self, layer: int, k_new, v_new, stream=None) -> None:
        """Writes new tokens [bh, n, d] behind the residual of one layer (the
        library's append kernel on that layer alone; the cache's residual count
        is left as it is: call :meth:`advance` once every layer has its
        tokens)."""
        n = int(k_new.shape[1])
        if self.n_res + n > int(self.state.r_cap):
            raise ValueError("residual ring overflow")
        st = kivi_cache.from_buffer_copy(self.state)   # the count advances in the copy only
        kivi_append((kivi_layer * 1)(self.layers[layer]), 1, st, [k_new], [v_new], n,
                    stream=stream)

    def advance(self, n: int) -> None:
        if self.n_res + n > int(self.state.r_cap):
            raise ValueError("residual ring overflow")
        self.state.n_res += n

    def append_flush(self, k_new, v_new, stream=None) -> int:
        """New tokens of every layer (fp16 [n_layers, bh, n, d] or per-layer
        lists of [bh, n, d], one bh stride) behind the residual, then the
        flush, in one call; returns the tokens flushed."""
        ks = list(k_new.unbind(0)) if hasattr(k_new, "unbind") else list(k_new)
        vs = list(v_new.unbind(0)) if hasattr(v_new, "unbind") else list(v_new)
        for x in ks + vs:
            _fp16_3d(x, "append_flush")
            if _bh_stride(x) != _bh_stride(ks[0]):
                raise ValueError("append_flush: every new-token tensor needs the same bh stride")
        return kivi_append_flush(self.layers, self.n_layers, self.state, ks, vs,
                                 int(ks[0].shape[1]), _bh_stride(ks[0]), stream)

    def append_all(self, k_new, v_new, stream=None) -> None:
        """New tokens of every layer (fp16 [n_layers, bh, n, d] tensors or
        per-layer lists of [bh, n, d]) behind the residual, in one launch; the
        residual count advances by n."""
        ks = list(k_new.unbind(0)) if hasattr(k_new, "unbind") else list(k_new)
        vs = list(v_new.unbind(0)) if hasattr(v_new, "unbind") else list(v_new)
        kivi_append(self.layers, self.n_layers, self.state, ks, vs, int(ks[0].shape[1]),
                    stream=stream)

    # hot path --------------------------------------------------------------
    def flush(self, stream=None, events=None) -> int:
        return kivi_flush(self.layers, self.n_layers, self.state, stream, events)

    def flush_fakequant(self, stream=None, events=None) -> int:
        """Flush that also writes the fp16 reconstruction of the flushed tokens
        into ``k_hat``/``v_hat`` (needs ``recon=True``)."""
        if not self.recon:
            raise ValueError("flush_fakequant needs a cache built with recon=True")
        return kivi_flush_fakequant(self.layers, self.n_layers, self.state, self._k_hat_ptrs,
                                    self._v_hat_ptrs, stream, events)

    def decode_attention(self, q, batch: int, sm_scale: Optional[float] = None, out=None,
                         n_split: Optional[int] = None, workspace=None, stream=None,
                         sinks: Optional["KiviSinks"] = None):
        """Attention of the new query tokens over everything the cache holds
        (packed store + fp16 residual; with ``sinks``, the stored sinks' fp16
        rows in place of their store slots).  ``q``: fp16 [n_layers, batch,
        h_q, d] (or a per-layer list); returns fp32 [n_layers, batch, h_q, d]."""
        import math
        import torch
        qs = list(q.unbind(0)) if hasattr(q, "unbind") else list(q)
        h_q, d = int(qs[0].shape[1]), int(qs[0].shape[2])
        if out is None:
            out = torch.empty((self.n_layers, batch, h_q, d), dtype=torch.float32,
                              device=qs[0].device)
        outs = list(out.unbind(0)) if hasattr(out, "unbind") else list(out)
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(d)
        if n_split is None:
            n_split = kivi_decode_attention_splits(self.state, self.n_layers, batch)
        if n_split > 1 and workspace is None:
            need = kivi_decode_attention_workspace(self.state, self.n_layers, batch, h_q, n_split)
            workspace = torch.empty(max(need, 1), dtype=torch.float32, device=qs[0].device)
        if sinks is None:
            kivi_decode_attention(self.layers, self.n_layers, self.state, batch, h_q, sm_scale,
                                  qs, outs, n_split, workspace, stream)
        else:
            kivi_decode_attention_sinks(self.layers, sinks.layers, self.n_layers, self.state,
                                        sinks.cfg, batch, h_q, sm_scale, qs, outs, n_split,
                                        workspace, stream)
        return out

    def dequantize(self, k_out=None, v_out=None, stream=None, events=None):
        """fp16 reconstructions of the first s_q store tokens of every layer;
        ``k_out``/``v_out`` default to new [n_layers, bh, s_q, d] tensors
        (returned as per-layer lists)."""
        import torch
        bh, d, s = int(self.state.bh), int(self.state.d), self.s_q
        dev = self.k_res[0].device
        if k_out is None:
            k_out = list(torch.empty((self.n_layers, bh, s, d), dtype=torch.float16,
                                     device=dev).unbind(0))
        if v_out is None:
            v_out = list(torch.empty((self.n_layers, bh, s, d), dtype=torch.float16,
                                     device=dev).unbind(0))
        kivi_dequantize_cache(self.layers, self.n_layers, self.state, k_out, v_out, stream,
                              events)
        return k_out, v_out


# ---------------------------------------------------------------------------
# KIVI-Sink
# ---------------------------------------------------------------------------

def kivi_sink_update(layers, sinks, n_layers: int, cache: kivi_cache, cfg: kivi_sink_cfg,
                     i0: int, n: int, stream=None) -> None:
    _check(lib().kivi_sink_update(layers, sinks, n_layers, C.byref(cache), C.byref(cfg), i0, n,
                                  _stream_handle(stream)), "kivi_sink_update")


def kivi_flush_sink(layers, sinks, n_layers: int, cache: kivi_cache, cfg: kivi_sink_cfg,
                    stream=None) -> int:
    n = C.c_int64(0)
    _check(lib().kivi_flush_sink(layers, sinks, n_layers, C.byref(cache), C.byref(cfg),
                                 C.byref(n), _stream_handle(stream)), "kivi_flush_sink")
    return int(n.value)


def kivi_sink_restore(sinks, n_layers: int, cache: kivi_cache, cfg: kivi_sink_cfg, k_out, v_out,
                      stream=None) -> None:
    _check(lib().kivi_sink_restore(sinks, n_layers, C.byref(cache), C.byref(cfg),
                                   _ptr_array(k_out, n_layers), _ptr_array(v_out, n_layers),
                                   _stream_handle(stream)), "kivi_sink_restore")


class KiviSinks:
    """KIVI-Sink state of every layer of a :class:`KiviCache` (device tensors):
    running top-k positions and scores, the sink store (positions and fp16
    key / value rows) and the flush's mask scratch."""

    def __init__(self, cache: "KiviCache", batch: int, k_top: int, sink_cap: int):
        import torch
        st = cache.state
        L, bh, d, r_cap = cache.n_layers, int(st.bh), int(st.d), int(st.r_cap)
        dev = cache.k_res[0].device
        self.cache, self.batch, self.k_top, self.sink_cap = cache, batch, k_top, sink_cap
        z = lambda shape, dt: torch.zeros((L,) + shape, dtype=dt, device=dev)  # noqa: E731
        kt, sc = max(k_top, 1), max(sink_cap, 1)
        self.top_pos = z((batch, kt), torch.int64)
        self.top_score = z((batch, kt), torch.float32)
        self.top_count = z((batch,), torch.int32)
        self.sink_pos = z((batch, sc), torch.int64)
        self.sink_count = z((batch,), torch.int32)
        self.sink_k = z((bh, sc, d), torch.float16)
        self.sink_v = z((bh, sc, d), torch.float16)
        self.mask = z((batch, (r_cap + 31) // 32), torch.int32)
        self.scores = z((batch, r_cap), torch.float32)
        self.layers = (kivi_sink_layer * L)(*[
            kivi_sink_layer(self.top_pos[i].data_ptr(), self.top_score[i].data_ptr(),
                            self.top_count[i].data_ptr(), self.sink_pos[i].data_ptr(),
                            self.sink_count[i].data_ptr(), self.sink_k[i].data_ptr(),
                            self.sink_v[i].data_ptr(), self.mask[i].data_ptr(),
                            self.scores[i].data_ptr())
            for i in range(L)])
        self.cfg = kivi_sink_cfg(batch, k_top, sink_cap, 0, 0)

    def update(self, i0: int, n: int, stream=None) -> None:
        """Score residual tokens i0 .. i0+n-1 and merge them into the top-k."""
        c = self.cache
        kivi_sink_update(c.layers, self.layers, c.n_layers, c.state, self.cfg, i0, n, stream)

    def flush(self, stream=None) -> int:
        c = self.cache
        return kivi_flush_sink(c.layers, self.layers, c.n_layers, c.state, self.cfg, stream)

    def restore(self, k_out, v_out, stream=None) -> None:
        c = self.cache
        kivi_sink_restore(self.layers, c.n_layers, c.state, self.cfg, k_out, v_out, stream)
