"""Seeded synthetic KV-cache workloads (inputs only, no quantizer arithmetic).

The shapes follow the models the KIVI pages measured (VeloxQuant-MLX blog post
"How I fused KIVI's KV-cache quantization into two bit-exact Metal kernels",
sections "Generation 1" and "Generation 4": Llama-3.2-3B 28 layers x 8 KV
heads x head_dim 128, Qwen2.5-7B 28 layers x 4 KV heads, Mistral-7B 32 layers
x 8 KV heads; KIVI defaults 2 bits, group 32, residual 32).  The pages'
models, prompts and results files are not available; these tensors stand in
for their keys and values.

Each element is a pure function of (seed, tensor, bh, token, channel), drawn
by the C generator ``kivi_inputs.c`` (counter-based, thread-count invariant).
``seed`` is the workload's index in :data:`CONFIGS`; ``tensor`` is
``layer * 2 + (0 for keys, 1 for values)``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_inputs.c")
_LIB = os.path.join(_HERE, "_build", "libkivi_inputs.so")

NORMAL, STUDENT_T, LAPLACE = 0, 1, 2


class _Spec(C.Structure):
    _fields_ = [("seed", C.c_uint64), ("tensor", C.c_uint64), ("dist", C.c_int32),
                ("nu", C.c_int32), ("sigma", C.c_double), ("heads", C.c_int32),
                ("n_outliers", C.c_int32), ("outlier_mult", C.c_double),
                ("fixed_outliers", C.POINTER(C.c_int32)), ("offset_amp", C.c_double)]


@dataclass(frozen=True)
class Dist:
    """Distribution of one tensor kind (keys or values)."""
    kind: int = NORMAL
    sigma: float = 1.0
    nu: int = 4
    n_outliers: int = 0
    outlier_mult: float = 1.0
    fixed_outliers: Tuple[int, ...] = ()
    offset_amp: float = 0.0


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: int
    batch: int
    kv_heads: int
    seq: int              # tokens per sequence in the residual / tensor
    head_dim: int
    bits: int
    group: int
    residual: int
    keys: Dist
    values: Dist
    # batched decode only: store tokens already present, new tokens per step, steps
    store_prefill: int = 0
    new_per_step: int = 0
    steps: int = 0
    sweep_bits: Tuple[int, ...] = ()
    sweep_groups: Tuple[int, ...] = ()
    note: str = ""

    @property
    def bh(self) -> int:
        return self.batch * self.kv_heads


_KEY_OUTLIERS_4x15 = Dist(NORMAL, 1.0, n_outliers=4, outlier_mult=15.0)

CONFIGS = {
    "tiny_flush": Workload(
        "tiny_flush", 0, layers=1, batch=1, kv_heads=8, seq=128, head_dim=128,
        bits=2, group=32, residual=32,
        keys=Dist(NORMAL, 1.0, n_outliers=4, outlier_mult=15.0,
                  fixed_outliers=(3, 17, 64, 101), offset_amp=2.0),
        values=Dist(NORMAL, 1.0),
        note="B=1 H_kv=8 S=128 D=128; keys N(0,1), channels {3,17,64,101} x15, "
             "per (head, channel) offset U(-2,2); values N(0,1); 2-bit, G=32, R=32"),
    "llama3_2_3b_prefill": Workload(
        "llama3_2_3b_prefill", 1, layers=28, batch=1, kv_heads=8, seq=4096, head_dim=128,
        bits=2, group=32, residual=32, keys=_KEY_OUTLIERS_4x15, values=Dist(NORMAL, 1.0),
        note="28 layers x B=1 H_kv=8 S=4096 D=128; keys N(0,1) with 4/128 outlier "
             "channels x15 per head; values N(0,1); 2-bit, G=32, R=32"),
    "qwen2_5_7b_long": Workload(
        "qwen2_5_7b_long", 2, layers=28, batch=1, kv_heads=4, seq=32768, head_dim=128,
        bits=4, group=64, residual=64,
        keys=Dist(STUDENT_T, 1.0, nu=4, n_outliers=6, outlier_mult=20.0),
        values=Dist(NORMAL, 0.5),
        note="28 layers x B=1 H_kv=4 S=32768 D=128; keys Student-t(4) with 6 outlier "
             "channels x20; values N(0, sd 0.5); 4-bit, G=64, R=64"),
    "batched_decode": Workload(
        "batched_decode", 3, layers=32, batch=64, kv_heads=8, seq=64, head_dim=128,
        bits=2, group=32, residual=32, keys=_KEY_OUTLIERS_4x15, values=Dist(NORMAL, 1.0),
        store_prefill=2048, new_per_step=32, steps=100,
        note="32 layers x B=64 H_kv=8 D=128; 2-bit store of S=2048 per sequence; each "
             "step appends 32 tokens and flushes 32 (G=32, R=32); 100 steps"),
    "large_store_sweep": Workload(
        "large_store_sweep", 4, layers=1, batch=16, kv_heads=8, seq=16384, head_dim=128,
        bits=2, group=32, residual=0, keys=_KEY_OUTLIERS_4x15, values=Dist(LAPLACE, 1.0),
        sweep_bits=(2, 4, 8), sweep_groups=(32, 64, 128),
        note="B=16 H_kv=8 S=16384 D=128; keys N(0,1) + 4 outlier channels x15, values "
             "Laplace(0,1); bits {2,4,8} x G {32,64,128}; full quantize then dequantize"),
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    stale = not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc, "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", _SRC,
                        "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.kivi_gen_fill.argtypes = [C.POINTER(_Spec), C.c_void_p, C.c_int64, C.c_int64,
                                        C.c_int64, C.c_int64, C.c_int64, C.c_int]
            L.kivi_gen_fill.restype = C.c_int
            L.kivi_gen_fill_range.argtypes = [C.POINTER(_Spec), C.c_void_p, C.c_int64,
                                              C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                              C.c_int64, C.c_int]
            L.kivi_gen_fill_range.restype = C.c_int
            L.kivi_gen_outliers.argtypes = [C.POINTER(_Spec), C.c_int64, C.c_int,
                                            C.POINTER(C.c_int32)]
            L.kivi_gen_outliers.restype = C.c_int
            _lib = L
    return _lib


def _spec(w: Workload, layer: int, kind: str):
    dist = w.keys if kind == "k" else w.values
    fixed = None
    n_out = dist.n_outliers
    if dist.fixed_outliers:
        fixed = (C.c_int32 * len(dist.fixed_outliers))(*dist.fixed_outliers)
        n_out = len(dist.fixed_outliers)
    spec = _Spec(w.seed, layer * 2 + (0 if kind == "k" else 1), dist.kind, dist.nu,
                 dist.sigma, w.kv_heads, n_out, dist.outlier_mult,
                 fixed if fixed is not None else C.POINTER(C.c_int32)(), dist.offset_amp)
    return spec, fixed


def default_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def fill(w: Workload, layer: int, kind: str, out: np.ndarray, tok0: int = 0,
         n_threads: Optional[int] = None, bh0: int = 0) -> np.ndarray:
    """Fill ``out`` (uint16 [bh, n_tok, d] view, last two dims contiguous) with
    sequence positions ``tok0 .. tok0 + n_tok`` of (layer, kind), bh slices
    ``bh0 .. bh0 + bh``."""
    assert out.dtype == np.uint16 and out.ndim == 3
    bh, n_tok, d = out.shape
    assert out.strides[2] == 2 and out.strides[1] == 2 * d
    spec, keep = _spec(w, layer, kind)
    rc = _load().kivi_gen_fill_range(C.byref(spec), out.ctypes.data, bh0, bh, tok0, n_tok, d,
                                     out.strides[0] // 2, n_threads or default_threads())
    if rc != 0:
        raise ValueError("input generator rejected its arguments")
    del keep
    return out


def generate(w: Workload, layer: int, kind: str, tok0: int = 0, n_tok: Optional[int] = None,
             bh: Optional[int] = None, n_threads: Optional[int] = None,
             bh0: int = 0) -> np.ndarray:
    """uint16 [bh, n_tok, d] fp16 bit patterns of (layer, kind) at positions
    tok0.., bh slices bh0 .. bh0 + bh."""
    n_tok = w.seq if n_tok is None else n_tok
    bh = w.bh - bh0 if bh is None else bh
    out = np.empty((bh, n_tok, w.head_dim), np.uint16)
    return fill(w, layer, kind, out, tok0, n_threads, bh0)


def outlier_channels(w: Workload, layer: int, head: int) -> np.ndarray:
    spec, keep = _spec(w, layer, "k")
    n = spec.n_outliers
    out = (C.c_int32 * max(1, n))()
    if _load().kivi_gen_outliers(C.byref(spec), w.head_dim, head, out) != 0:
        raise ValueError("bad outlier query")
    del keep
    return np.array(out[:n], dtype=np.int64)


def custom(name: str = "custom", seed: int = 100, batch: int = 1, kv_heads: int = 2,
           seq: int = 96, head_dim: int = 128, bits: int = 2, group: int = 32,
           residual: int = 32, keys: Dist = _KEY_OUTLIERS_4x15,
           values: Dist = Dist(NORMAL, 1.0)) -> Workload:
    """A small workload of arbitrary shape for parity tests."""
    return Workload(name, seed, 1, batch, kv_heads, seq, head_dim, bits, group, residual,
                    keys, values)
