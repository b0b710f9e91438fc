#!/usr/bin/env python
"""Throughput of the KIVI KV-cache flush + dequantize path on one or more GPUs.

One step = one pass of the whole hot path over one batch of synthetic input:
for every layer, the flush of the fp16 residual window (keys quantized per
channel, values per token, codes bit-packed, scales/zeros written, flush
bookkeeping) followed by the dequantization of the store back to fp16.
The metric is HBM bandwidth in algorithmic bytes (bytes read + written by
the definition of the operation) per second:

    quantize   2 + b/8 + 8/G  bytes per fp16 element (read fp16, write codes,
                              scale and zero)
    dequantize b/8 + 8/G + 2  bytes per fp16 element

Default workload: 28 layers x 4 KV heads x 32768 tokens x head_dim 128
(Qwen2.5-7B shape, long context), 4-bit, G = 64, residual 64, so each layer
flushes 32704 tokens; one step moves ~4.9 GB.  The same line then carries the
nine (bits, G) cells of the large store sweep ([128 x 16384 x 128] keys and
values, full quantize then full dequantize; ``--no-sweep`` leaves them out),
each timed the same way.  Inputs are seeded synthetic tensors
(``workloads``), resident in HBM before the timed region; every kernel pass
moves more than the 129 MB L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle on the same metric

With ``--gpus N`` (N > 1) outside torchrun the script relaunches itself
under ``torch.distributed.run`` with N processes; under torchrun every rank
runs the same workload on its own GPU (independent shards, no collective on
the data path); the step time is the maximum over ranks and ``value`` counts
the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize+dequant HBM GB/s (bytes in+out) and % of GB300 HBM peak"
NOMINAL_HBM_GBS = 8000.0
DEFAULT_WORKLOAD = "qwen2_5_7b_long"
FALLBACK_HBM_GBS = 6800.0
# Kernel sources behind each kind of workload: a committed ncu traffic figure
# stays valid while these files hash to the value stored with it.
_COMMON_FILES = ("kivi_api.cu", "kivi_device.cuh", "kivi_arith.cuh", "kivi_launch.h",
                 "kivi_dispatch.h")
CSRC_FILES = {
    "flush": _COMMON_FILES + ("kivi_keys.cu", "kivi_values.cu", "kivi_staged.cu",
                              "kivi_ring.cu", "kivi_expand.cuh"),
    "attention": _COMMON_FILES + ("kivi_expand.cuh", "kivi_attention_kernel.cuh",
                                  "kivi_attention.cu", "kivi_attention_d64.cu",
                                  "kivi_attention_d256.cu", "kivi_tc_common.cuh",
                                  "kivi_attention_ws.cu"),
    "sink": _COMMON_FILES + ("kivi_keys.cu", "kivi_values.cu", "kivi_staged.cu",
                             "kivi_sink.cu", "kivi_expand.cuh"),
}


def spread_us(ms: list) -> dict:
    """Per-step times of one kernel (ms) -> median, min, max and the
    interquartile range relative to the median (the run-to-run noise of an
    unchanged kernel), in microseconds and percent."""
    v = sorted(ms)
    n = len(v)

    def q(f):                       # linear interpolation between order statistics
        x = f * (n - 1)
        i = int(x)
        return v[i] if i + 1 >= n else v[i] + (v[i + 1] - v[i]) * (x - i)

    med = q(0.5)
    return {"median_us": round(med * 1e3, 2), "min_us": round(v[0] * 1e3, 2),
            "max_us": round(v[-1] * 1e3, 2),
            "iqr_pct": round((q(0.75) - q(0.25)) / med * 100, 2) if med > 0 else None}


def host_cpu() -> dict:
    """Logical CPUs and the CPU model of the host (for the CPU baselines)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def e2e_bounds(layers: int, n_chunks: int, ramp=()) -> list:
    """Layer bounds of the end-to-end pipeline's chunks: about n_chunks equal
    chunks, the first of them split into the ramp's smaller sizes (the
    device-to-host copies, the longer direction, start once the first chunk
    is in and flushed)."""
    base = max(1, -(-layers // max(1, n_chunks)))
    bounds = [0]
    for r in ramp:
        if r >= base or bounds[-1] + r > layers:
            break
        bounds.append(bounds[-1] + r)
    rest = layers - bounds[-1]
    k = max(1, round(rest / base)) if rest > 0 else 0
    bounds += [bounds[-1] + rest * (i + 1) // k for i in range(k)]
    return bounds


def bytes_per_elem(bits: int, group: int) -> float:
    return 2.0 + bits / 8.0 + 8.0 / group


def fused_bytes_per_elem(bits: int, group: int) -> float:
    """Fused fake-quant pass: read fp16, write codes + scale + zero, write the
    fp16 reconstruction."""
    return 4.0 + bits / 8.0 + 8.0 / group


# ---------------------------------------------------------------------------
# distributed helpers (timing reduction only; the data path has no collective)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for name, flag in zip(names, p[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def pinned_u16(shape):
    import numpy as np
    import torch
    t = torch.empty(shape, dtype=torch.float16, pin_memory=True)
    return t, t.view(torch.int16).numpy().view(np.uint16)


class PrefillFlush:
    """All layers' residual rings hold the prompt; one step = flush (all
    layers, keys then values) + dequantization of the store (all layers)."""

    kernels = ("key_quant", "value_quant", "key_dequant", "value_dequant")
    events_per_step = 6

    def __init__(self, w, device):
        import ctypes as C
        import torch
        import kv_cache_quantization_kivi_gb300 as K
        import workloads as W
        self.w, self.K = w, K
        L, bh, S, d = w.layers, w.bh, w.seq, w.head_dim
        self.n = K.kivi_flush_size(S, w.residual, w.group)
        self.cache = K.KiviCache(L, bh, d, r_cap=S, cap=S, group=w.group, bits=w.bits,
                                 residual=w.residual, device=device)
        # host inputs in pinned memory (also the e2e source), generated in place
        self.k_host_t, self.k_host = pinned_u16((L, bh, S, d))
        self.v_host_t, self.v_host = pinned_u16((L, bh, S, d))
        for l in range(L):
            W.fill(w, l, "k", self.k_host[l])
            W.fill(w, l, "v", self.v_host[l])
        self.cache.k_res_all.copy_(self.k_host_t.to(device))
        self.cache.v_res_all.copy_(self.v_host_t.to(device))
        self.k_out = torch.empty((L, bh, self.n, d), dtype=torch.float16, device=device)
        self.v_out = torch.empty((L, bh, self.n, d), dtype=torch.float16, device=device)
        self.k_ptrs = (C.c_void_p * L)(*[t.data_ptr() for t in self.k_out.unbind(0)])
        self.v_ptrs = (C.c_void_p * L)(*[t.data_ptr() for t in self.v_out.unbind(0)])
        elems = L * bh * self.n * d
        bpe = bytes_per_elem(w.bits, w.group)
        self.kernel_bytes = {k: elems * bpe for k in self.kernels}
        self.step_bytes = 4 * elems * bpe
        self.step_elems = 2 * elems      # fp16 elements flushed (keys and values)
        self.launches_per_step = 4

    def config(self):
        w = self.w
        return {"workload": w.name, "layers": w.layers, "bh": w.bh, "seq": w.seq,
                "head_dim": w.head_dim, "bits": w.bits, "group": w.group,
                "residual": w.residual, "tokens_flushed_per_layer": self.n,
                "step": "flush (per-channel key + per-token value quantize, pack, bookkeeping) "
                        "+ dequantize of the store, all layers"}

    def step(self, stream, ev=None):
        c = self.cache
        c.reset(s_q=0, res_head=0, n_res=self.w.seq)
        n = c.flush(stream, None if ev is None else ev[0])
        assert n == self.n
        self.K.kivi_dequantize_cache(c.layers, c.n_layers, c.state, self.k_ptrs, self.v_ptrs,
                                     stream, None if ev is None else ev[1])

    def step_events(self, evs):
        """Event handles for one step from its events_per_step torch events."""
        return (self.K.event_handles(evs[0:3]), self.K.event_handles(evs[3:6]))

    def kernel_times(self, e):
        return {"key_quant": e[0].elapsed_time(e[1]), "value_quant": e[1].elapsed_time(e[2]),
                "key_dequant": e[3].elapsed_time(e[4]), "value_dequant": e[4].elapsed_time(e[5])}

    def e2e_setup(self):
        import torch
        L, bh, d = self.w.layers, self.w.bh, self.w.head_dim
        self.k_back = torch.empty((L, bh, self.n, d), dtype=torch.float16, pin_memory=True)
        self.v_back = torch.empty((L, bh, self.n, d), dtype=torch.float16, pin_memory=True)
        c = self.cache
        self.store_dev = [c.k_codes_all, c.k_scale_all, c.k_zero_all, c.v_codes_all,
                          c.v_scale_all, c.v_zero_all]
        self.store_back = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                           for t in self.store_dev]
        h2d = 2 * self.k_host_t.numel() * 2
        d2h = 2 * self.k_back.numel() * 2 + sum(t.numel() * t.element_size()
                                                for t in self.store_back)
        import ctypes as C
        # pipeline over layer chunks: the host-to-device copy of chunk i+1, the
        # kernels of chunk i and the device-to-host copy of chunk i-1 run at
        # once on three streams, ordered by events
        K = self.K
        device = c.k_res_all.device
        self.e2e_streams = (torch.cuda.Stream(device), torch.cuda.Stream(device))
        c.reset(s_q=0, res_head=0, n_res=self.w.seq)
        L = self.w.layers
        bounds = e2e_bounds(L, self.E2E_CHUNKS, self.E2E_RAMP)
        n_chunks = len(bounds) - 1
        self.e2e_chunks = []
        for l0, l1 in zip(bounds[:-1], bounds[1:]):
            n = l1 - l0
            self.e2e_chunks.append((l0, l1, (K.kivi_layer * n)(*c.layers[l0:l1]),
                                    (C.c_void_p * n)(*self.k_ptrs[l0:l1]),
                                    (C.c_void_p * n)(*self.v_ptrs[l0:l1]),
                                    K.kivi_cache.from_buffer_copy(c.state)))
        self.e2e_pipeline = (f"{n_chunks} chunks of layers; host-to-device copies, kernels and "
                             "device-to-host copies on three streams, captured once in a CUDA "
                             "graph and replayed every step")
        self.e2e_graph = None
        return h2d, d2h

    # measured end to end (GB/s, llama3_2_3b_prefill / qwen2_5_7b_long): 7
    # equal chunks 295 / 317, with a (1, 1, 2) ramp 301 / 325; 5 chunks with a
    # (1, 1, 2, 2) ramp 303 / 178 (the 5.5-layer chunks of the long prompt
    # copy slowly)
    E2E_CHUNKS = 7
    E2E_RAMP = (1, 1, 2)

    def e2e_step(self, stream):
        import torch
        if self.e2e_graph is None:
            # capture the pipelined step (the library's C-ABI calls and the copies
            # on three streams) once; every step replays it on `stream`
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(stream.device)
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                self._e2e_issue(cap)
            stream.wait_stream(cap)
            self.e2e_graph = g
        self.e2e_graph.replay()

    def _e2e_issue(self, stream):
        import torch
        K = self.K
        c = self.cache
        s_in, s_out = self.e2e_streams
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for l0, l1, layers, kp, vp, state0 in self.e2e_chunks:
            with torch.cuda.stream(s_in):
                c.k_res_all[l0:l1].copy_(self.k_host_t[l0:l1], non_blocking=True)
                c.v_res_all[l0:l1].copy_(self.v_host_t[l0:l1], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            st = K.kivi_cache.from_buffer_copy(state0)
            assert K.kivi_flush(layers, l1 - l0, st, stream) == self.n
            K.kivi_dequantize_cache(layers, l1 - l0, st, kp, vp, stream)
            ev_done = torch.cuda.Event()
            ev_done.record(stream)
            s_out.wait_event(ev_done)
            with torch.cuda.stream(s_out):
                self.k_back[l0:l1].copy_(self.k_out[l0:l1], non_blocking=True)
                self.v_back[l0:l1].copy_(self.v_out[l0:l1], non_blocking=True)
                for dst, src in zip(self.store_back, self.store_dev):
                    dst[l0:l1].copy_(src[l0:l1], non_blocking=True)
        end = torch.cuda.Event()
        end.record(s_out)
        stream.wait_event(end)

    def cpu_sample(self, budget_s: float):
        """The oracle on whole layers of the same workload until the budget is spent."""
        import oracle as O
        w = self.w
        done_bytes, t_total, layers = 0.0, 0.0, 0
        elems = w.bh * self.n * w.head_dim
        W_ = 32 // w.bits
        t_fn = {"flush": 0.0, "dequantize_keys": 0.0, "dequantize_values": 0.0}
        for l in range(w.layers):
            st = O.Store(w.bh, w.head_dim, w.seq, w.group, w.bits)
            k, v = self.k_host[l], self.v_host[l]
            t0 = time.perf_counter()
            n, _, _, _ = O.flush(k, v, st, w.residual, 0, 0, w.seq)
            t1 = time.perf_counter()
            O.dequantize_keys(st.k_codes[:, :n // W_], st.k_scale[:, :n // w.group],
                              st.k_zero[:, :n // w.group], n, w.group, w.bits)
            t2 = time.perf_counter()
            O.dequantize_values(st.v_codes[:, :n], st.v_scale[:, :n], st.v_zero[:, :n],
                                w.group, w.bits)
            t3 = time.perf_counter()
            t_fn["flush"] += t1 - t0
            t_fn["dequantize_keys"] += t2 - t1
            t_fn["dequantize_values"] += t3 - t2
            t_total += t3 - t0
            done_bytes += 4 * elems * bytes_per_elem(w.bits, w.group)
            layers += 1
            if t_total >= budget_s:
                break
        per_fn = ", ".join(f"{k} {v / layers * 1e3:.0f} ms" for k, v in t_fn.items())
        return done_bytes, t_total, (f"{layers} of {w.layers} layers (flush + dequantize, keys "
                                     f"and values; per layer: {per_fn})")


class SinkPrefillFlush(PrefillFlush):
    """The prefill flush with KIVI-Sink protection: every prompt token's key
    norm is scored and ranked (top 5 per sequence), the flush keeps the
    flushed top-5 tokens fp16 in the sink store and out of the groups'
    min/max, and the dequantized store gets the sinks' rows back."""

    kernels = ("sink_update", "flush_sink", "dequantize", "sink_restore")
    events_per_step = 5
    K_TOP = 5

    def __init__(self, w, device):
        super().__init__(w, device)
        K = self.K
        self.sinks = K.KiviSinks(self.cache, w.batch, self.K_TOP, 2 * self.K_TOP)
        elems = w.layers * w.bh * self.n * w.head_dim
        score_bytes = w.layers * w.bh * w.seq * w.head_dim * 2        # the prompt's keys read
        bpe = bytes_per_elem(w.bits, w.group)
        self.kernel_bytes = {"sink_update": score_bytes, "flush_sink": 2 * elems * bpe,
                             "dequantize": 2 * elems * bpe, "sink_restore": 0.0}
        self.step_bytes = score_bytes + 4 * elems * bpe
        self.launches_per_step = 8
        self.k_list = list(self.k_out.unbind(0))
        self.v_list = list(self.v_out.unbind(0))

    def config(self):
        c = super().config()
        c["step"] = ("KIVI-Sink: key-norm scores and top-5 of every prompt token, sink-protected "
                     "flush (mask, quantize, sink store), dequantize of the store, sinks restored")
        c["k_top"] = self.K_TOP
        return c

    def step(self, stream, ev=None):
        c, sk = self.cache, self.sinks
        sk.top_count.zero_()
        sk.sink_count.zero_()
        c.reset(s_q=0, res_head=0, n_res=self.w.seq)
        if ev is not None:
            ev[0].record(stream)
        sk.update(0, self.w.seq, stream)
        if ev is not None:
            ev[1].record(stream)
        n = sk.flush(stream)
        assert n == self.n
        if ev is not None:
            ev[2].record(stream)
        self.K.kivi_dequantize_cache(c.layers, c.n_layers, c.state, self.k_ptrs, self.v_ptrs,
                                     stream)
        if ev is not None:
            ev[3].record(stream)
        sk.restore(self.k_list, self.v_list, stream)
        if ev is not None:
            ev[4].record(stream)

    def step_events(self, evs):
        return evs

    def kernel_times(self, e):
        return {"sink_update": e[0].elapsed_time(e[1]), "flush_sink": e[1].elapsed_time(e[2]),
                "dequantize": e[2].elapsed_time(e[3]), "sink_restore": e[3].elapsed_time(e[4])}

    def cpu_sample(self, budget_s: float):
        import oracle as O
        w = self.w
        done, t_total, layers = 0.0, 0.0, 0
        W_ = 32 // w.bits
        per_layer = self.step_bytes / w.layers
        for l in range(w.layers):
            st = O.Store(w.bh, w.head_dim, w.seq, w.group, w.bits)
            ss = O.SinkState(w.batch, w.kv_heads, w.head_dim, self.K_TOP, 2 * self.K_TOP)
            k, v = self.k_host[l], self.v_host[l]
            t0 = time.perf_counter()
            ss.update(O.sink_scores(k, w.kv_heads), 0)
            n, _, _, _ = O.flush_sink(k, v, st, w.residual, 0, 0, w.seq, ss)
            ky = O.dequantize_keys(st.k_codes[:, :n // W_], st.k_scale[:, :n // w.group],
                                   st.k_zero[:, :n // w.group], n, w.group, w.bits)
            vy = O.dequantize_values(st.v_codes[:, :n], st.v_scale[:, :n], st.v_zero[:, :n],
                                     w.group, w.bits)
            O.sink_restore(ky, vy, ss)
            t_total += time.perf_counter() - t0
            done += per_layer
            layers += 1
            if t_total >= budget_s:
                break
        return done, t_total, f"{layers} of {w.layers} layers (KIVI-Sink score, flush, dequantize, restore)"

    def e2e_setup(self):
        return super().e2e_setup()


class FusedPrefillFlush(PrefillFlush):
    """The prefill flush in its fused fake-quant form: one launch per tensor
    kind over all layers quantizes the flushed tokens into the store and
    writes their fp16 reconstruction in the same pass (no dequantize pass
    re-reading the codes)."""

    kernels = ("key_fakequant", "value_fakequant")
    events_per_step = 3

    def __init__(self, w, device):
        import torch
        import kv_cache_quantization_kivi_gb300 as K
        import workloads as W
        self.w, self.K = w, K
        L, bh, S, d = w.layers, w.bh, w.seq, w.head_dim
        self.n = K.kivi_flush_size(S, w.residual, w.group)
        self.cache = K.KiviCache(L, bh, d, r_cap=S, cap=S, group=w.group, bits=w.bits,
                                 residual=w.residual, device=device, recon=True)
        self.k_host_t, self.k_host = pinned_u16((L, bh, S, d))
        self.v_host_t, self.v_host = pinned_u16((L, bh, S, d))
        for l in range(L):
            W.fill(w, l, "k", self.k_host[l])
            W.fill(w, l, "v", self.v_host[l])
        self.cache.k_res_all.copy_(self.k_host_t.to(device))
        self.cache.v_res_all.copy_(self.v_host_t.to(device))
        elems = L * bh * self.n * d
        bpe = fused_bytes_per_elem(w.bits, w.group)
        self.kernel_bytes = {k: elems * bpe for k in self.kernels}
        self.step_bytes = 2 * elems * bpe
        self.step_elems = 2 * elems
        self.launches_per_step = 2

    def config(self):
        c = super().config()
        c["step"] = ("fused fake-quant flush: per-channel key + per-token value quantize, "
                     "pack, bookkeeping and the fp16 reconstruction in one pass, all layers")
        c["bytes_per_elem"] = fused_bytes_per_elem(self.w.bits, self.w.group)
        return c

    def step(self, stream, ev=None):
        c = self.cache
        c.reset(s_q=0, res_head=0, n_res=self.w.seq)
        n = c.flush_fakequant(stream, ev)
        assert n == self.n

    def step_events(self, evs):
        return self.K.event_handles(evs[0:3])

    def kernel_times(self, e):
        return {"key_fakequant": e[0].elapsed_time(e[1]),
                "value_fakequant": e[1].elapsed_time(e[2])}

    def e2e_setup(self):
        import torch
        c, n = self.cache, self.n
        self.hat_dev = [c.k_hat_all[:, :, :n], c.v_hat_all[:, :, :n]]
        self.store_dev = [c.k_codes_all, c.k_scale_all, c.k_zero_all, c.v_codes_all,
                          c.v_scale_all, c.v_zero_all]
        self.back = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                     for t in self.hat_dev + self.store_dev]
        h2d = 2 * self.k_host_t.numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in self.back)
        return h2d, d2h

    def e2e_step(self, stream):
        c = self.cache
        c.k_res_all.copy_(self.k_host_t, non_blocking=True)
        c.v_res_all.copy_(self.v_host_t, non_blocking=True)
        self.step(stream)
        for dst, src in zip(self.back, self.hat_dev + self.store_dev):
            dst.copy_(src, non_blocking=True)

    def cpu_sample(self, budget_s: float):
        """The oracle (flush, then dequantization of the flushed tokens) on whole
        layers, counted in the fused pass's bytes."""
        import oracle as O
        w = self.w
        done_bytes, t_total, layers = 0.0, 0.0, 0
        elems = w.bh * self.n * w.head_dim
        W_ = 32 // w.bits
        for l in range(w.layers):
            st = O.Store(w.bh, w.head_dim, w.seq, w.group, w.bits)
            t0 = time.perf_counter()
            n, _, _, _ = O.flush(self.k_host[l], self.v_host[l], st, w.residual, 0, 0, w.seq)
            O.dequantize_keys(st.k_codes[:, :n // W_], st.k_scale[:, :n // w.group],
                              st.k_zero[:, :n // w.group], n, w.group, w.bits)
            O.dequantize_values(st.v_codes[:, :n], st.v_scale[:, :n], st.v_zero[:, :n],
                                w.group, w.bits)
            t_total += time.perf_counter() - t0
            done_bytes += 2 * elems * fused_bytes_per_elem(w.bits, w.group)
            layers += 1
            if t_total >= budget_s:
                break
        return done_bytes, t_total, (f"{layers} of {w.layers} layers (flush + dequantize of the "
                                     "flushed tokens, keys and values)")


class DecodeFlush:
    """Batched decode: every layer's store already holds 2048 tokens per
    sequence and its residual ring (2R = 64 rows) the R = 32 newest tokens;
    one step appends the next 32 tokens of every layer (keys and values,
    written behind the residual by the library's append) and flushes the 32
    oldest into the store, so the residual is back at R.  The store offset
    cycles over 100 consecutive flushes; the new tokens come from two
    device-resident sets used alternately."""

    kernels = ("append", "key_quant", "value_quant")
    events_per_step = 4
    RECON = False

    def __init__(self, w, device):
        import torch
        import kv_cache_quantization_kivi_gb300 as K
        import workloads as W
        self.w, self.K = w, K
        L, bh, d, G, R = w.layers, w.bh, w.head_dim, w.group, w.residual
        n = w.new_per_step
        self.r_cap = 2 * R
        self.cycle = w.steps
        cap = w.store_prefill + n * self.cycle
        self.cache = K.KiviCache(L, bh, d, r_cap=self.r_cap, cap=cap, group=G, bits=w.bits,
                                 residual=R, device=device, recon=self.RECON)
        # the ring's residual (tokens 2048 .. 2048+R-1) and two sets of new tokens
        self.k_host_t, self.k_host = pinned_u16((L, bh, self.r_cap, d))
        self.v_host_t, self.v_host = pinned_u16((L, bh, self.r_cap, d))
        for l in range(L):
            W.fill(w, l, "k", self.k_host[l], tok0=w.store_prefill)
            W.fill(w, l, "v", self.v_host[l], tok0=w.store_prefill)
        self.cache.k_res_all[:, :, :R].copy_(self.k_host_t[:, :, :R].to(device))
        self.cache.v_res_all[:, :, :R].copy_(self.v_host_t[:, :, :R].to(device))
        # new-token sets: set 0 = tokens 2048+R .., set 1 = tokens 2048+2R ..
        self.new_host, self.new_host_u16 = [], []
        for s in range(2):
            kt, kh = pinned_u16((L, bh, n, d))
            vt, vh = pinned_u16((L, bh, n, d))
            for l in range(L):
                W.fill(w, l, "k", kh[l], tok0=w.store_prefill + R + s * n)
                W.fill(w, l, "v", vh[l], tok0=w.store_prefill + R + s * n)
            self.new_host.append((kt, vt))
            self.new_host_u16.append((kh, vh))
        self.new_dev = [(kt.to(device), vt.to(device)) for kt, vt in self.new_host]
        self.new_ptrs = [(K._ptr_array(list(kd.unbind(0)), L), K._ptr_array(list(vd.unbind(0)), L))
                         for kd, vd in self.new_dev]
        self.new_bh_stride = n * d
        self.cache.reset(s_q=w.store_prefill, res_head=0, n_res=R)
        self.i = 0
        elems = L * bh * n * d
        bpe = (fused_bytes_per_elem if self.RECON else bytes_per_elem)(w.bits, G)
        qk = "key_fakequant" if self.RECON else "key_quant"
        qv = "value_fakequant" if self.RECON else "value_quant"
        # append: read the new fp16 tokens, write them into the ring (keys and values)
        self.kernel_bytes = {"append": 2 * elems * 4.0, qk: elems * bpe, qv: elems * bpe}
        self.step_bytes = sum(self.kernel_bytes.values())
        self.step_elems = 2 * elems
        self.launches_per_step = 3

    def config(self):
        w = self.w
        return {"workload": w.name, "layers": w.layers, "bh": w.bh, "head_dim": w.head_dim,
                "bits": w.bits, "group": w.group, "residual": w.residual,
                "store_tokens": w.store_prefill, "tokens_appended_per_step": w.new_per_step,
                "tokens_flushed_per_step": w.new_per_step,
                "consecutive_flushes": self.cycle,
                "residual_compaction_bytes_per_step": 0,
                "residual_storage": "a ring of 2R rows: the append writes behind the residual, "
                                    "the flush advances its head, nothing is copied",
                "step": "one decode step of every layer: append of the new tokens (keys and "
                        "values) and the flush of the oldest residual tokens",
                "bytes": "append 8 B per new fp16 element pair (read + ring write, K and V); "
                         "flush 2 + b/8 + 8/G per element"}

    def step(self, stream, ev=None):
        w, c = self.w, self.cache
        if self.i % self.cycle == 0:     # the store offset cycles; the ring runs on
            c.state.s_q = w.store_prefill
        kp, vp = self.new_ptrs[self.i % 2]
        self.i += 1
        self._append_flush(stream, kp, vp, ev)

    def _append_flush(self, stream, kp, vp, ev):
        # one call: the flush's launches overlap the append's tail
        w, c = self.w, self.cache
        n = self.K.kivi_append_flush(c.layers, c.n_layers, c.state, kp, vp, w.new_per_step,
                                     self.new_bh_stride, stream, ev)
        assert n == w.new_per_step

    def step_events(self, evs):
        return (C_void_p_array(evs))

    def kernel_times(self, e):
        names = self.kernels
        return {names[0]: e[0].elapsed_time(e[1]), names[1]: e[1].elapsed_time(e[2]),
                names[2]: e[2].elapsed_time(e[3])}

    def e2e_setup(self):
        import torch
        w = self.w
        # per step: the new tokens of every layer in, the flushed store slice out
        L, bh, d, G = w.layers, w.bh, w.head_dim, w.group
        n = w.new_per_step
        Wd = 32 // w.bits
        self.back = [torch.empty((L, bh, n // Wd, d), dtype=torch.int32, pin_memory=True),
                     torch.empty((L, bh, n // G, d), dtype=torch.float32, pin_memory=True),
                     torch.empty((L, bh, n // G, d), dtype=torch.float32, pin_memory=True),
                     torch.empty((L, bh, n, d // Wd), dtype=torch.int32, pin_memory=True),
                     torch.empty((L, bh, n, d // G), dtype=torch.float32, pin_memory=True),
                     torch.empty((L, bh, n, d // G), dtype=torch.float32, pin_memory=True)]
        h2d = 2 * self.new_host[0][0].numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in self.back)
        return h2d, d2h

    def _store_slices(self, s_q):
        c, w = self.cache, self.w
        n, G, Wd = w.new_per_step, w.group, 32 // w.bits
        return [c.k_codes_all[:, :, s_q // Wd:(s_q + n) // Wd],
                c.k_scale_all[:, :, s_q // G:(s_q + n) // G],
                c.k_zero_all[:, :, s_q // G:(s_q + n) // G], c.v_codes_all[:, :, s_q:s_q + n],
                c.v_scale_all[:, :, s_q:s_q + n], c.v_zero_all[:, :, s_q:s_q + n]]

    def e2e_step(self, stream):
        w, c = self.w, self.cache
        s = self.i % 2
        self.new_dev[s][0].copy_(self.new_host[s][0], non_blocking=True)
        self.new_dev[s][1].copy_(self.new_host[s][1], non_blocking=True)
        s_q = w.store_prefill if self.i % self.cycle == 0 else c.s_q
        self.step(stream)
        for dst, src in zip(self.back, self._store_slices(s_q)):
            dst.copy_(src, non_blocking=True)

    def cpu_sample(self, budget_s: float):
        import oracle as O
        w = self.w
        done, t_total, layers = 0.0, 0.0, 0
        cap = w.store_prefill + w.new_per_step
        R, n = w.residual, w.new_per_step
        per_layer = self.step_bytes / w.layers
        for l in range(w.layers):
            st = O.Store(w.bh, w.head_dim, cap, w.group, w.bits)
            k_ring = np.ascontiguousarray(self.k_host[l])
            v_ring = np.ascontiguousarray(self.v_host[l])
            kn, vn = self.new_host_u16[0][0][l], self.new_host_u16[0][1][l]
            t0 = time.perf_counter()
            n_res = O.append(k_ring, v_ring, 0, R, kn, vn)
            m, _, _, _ = O.flush(k_ring, v_ring, st, R, w.store_prefill, 0, n_res)
            t_total += time.perf_counter() - t0
            assert m == n
            done += per_layer
            layers += 1
            if t_total >= budget_s:
                break
        return done, t_total, (f"{layers} of {w.layers} layers (one decode step: append + "
                               "flush, keys and values)")


class FusedDecodeFlush(DecodeFlush):
    """The batched decode step in its fused fake-quant form: the append, then
    a flush that quantizes the 32 oldest residual tokens of every layer into
    the store and writes their fp16 reconstruction into the fp16 cache
    [bh, cap, d] in the same pass."""

    kernels = ("append", "key_fakequant", "value_fakequant")
    RECON = True

    def config(self):
        c = super().config()
        c["step"] = ("one fused fake-quant decode step of every layer: append of the new tokens, "
                     "then store and fp16 reconstruction of the flushed tokens in one pass")
        c["bytes_per_elem"] = fused_bytes_per_elem(self.w.bits, self.w.group)
        return c

    def _append_flush(self, stream, kp, vp, ev):
        # the fused flush has no combined call: append, then the flush
        w, c = self.w, self.cache
        if ev is not None:
            ev_torch, handles = ev
            ev_torch.record(stream)
        self.K.kivi_append(c.layers, c.n_layers, c.state, kp, vp, w.new_per_step,
                           new_bh_stride=self.new_bh_stride, stream=stream)
        n = c.flush_fakequant(stream, None if ev is None else handles)
        assert n == w.new_per_step

    def step_events(self, evs):
        return (evs[0], self.K.event_handles(evs[1:4]))

    def e2e_setup(self):
        import torch
        h2d, d2h = super().e2e_setup()
        w = self.w
        shape = (w.layers, w.bh, w.new_per_step, w.head_dim)
        self.hat_back = [torch.empty(shape, dtype=torch.float16, pin_memory=True)
                         for _ in range(2)]
        return h2d, d2h + sum(t.numel() * 2 for t in self.hat_back)

    def e2e_step(self, stream):
        w, c = self.w, self.cache
        n = w.new_per_step
        s_q = w.store_prefill if self.i % self.cycle == 0 else c.s_q
        super().e2e_step(stream)
        self.hat_back[0].copy_(c.k_hat_all[:, :, s_q:s_q + n], non_blocking=True)
        self.hat_back[1].copy_(c.v_hat_all[:, :, s_q:s_q + n], non_blocking=True)

    def cpu_sample(self, budget_s: float):
        import oracle as O
        w = self.w
        done, t_total, layers = 0.0, 0.0, 0
        cap = w.store_prefill + w.new_per_step
        Wd = 32 // w.bits
        s0, R = w.store_prefill, w.residual
        per_layer = self.step_bytes / w.layers
        for l in range(w.layers):
            st = O.Store(w.bh, w.head_dim, cap, w.group, w.bits)
            k_ring = np.ascontiguousarray(self.k_host[l])
            v_ring = np.ascontiguousarray(self.v_host[l])
            kn, vn = self.new_host_u16[0][0][l], self.new_host_u16[0][1][l]
            t0 = time.perf_counter()
            n_res = O.append(k_ring, v_ring, 0, R, kn, vn)
            n, _, _, _ = O.flush(k_ring, v_ring, st, R, s0, 0, n_res)
            O.dequantize_keys(st.k_codes[:, s0 // Wd:(s0 + n) // Wd],
                              st.k_scale[:, s0 // w.group:(s0 + n) // w.group],
                              st.k_zero[:, s0 // w.group:(s0 + n) // w.group], n, w.group, w.bits)
            O.dequantize_values(st.v_codes[:, s0:s0 + n], st.v_scale[:, s0:s0 + n],
                                st.v_zero[:, s0:s0 + n], w.group, w.bits)
            t_total += time.perf_counter() - t0
            done += per_layer
            layers += 1
            if t_total >= budget_s:
                break
        return done, t_total, (f"{layers} of {w.layers} layers (one decode step: append + flush "
                               "+ dequantize of the flushed tokens, keys and values)")


class DecodeAttention:
    """Decode attention over the batched-decode cache: every layer's store
    holds the first 2048 tokens of each sequence (quantized from the
    workload's data), the residual ring the next 64 in fp16; one step = one
    new query token per sequence and query head (32 query heads over the 8 KV
    heads) attending to all 2112 cached tokens of every layer, reading the
    packed codes directly."""

    kernels = ("decode_attention",)
    events_per_step = 2
    H_Q = 32

    def __init__(self, w, device):
        import numpy as np
        import torch
        import kv_cache_quantization_kivi_gb300 as K
        import workloads as W
        self.w, self.K = w, K
        L, bh, d, G, b = w.layers, w.bh, w.head_dim, w.group, w.bits
        n = w.store_prefill
        self.r_cap = 2 * w.residual
        self.cache = K.KiviCache(L, bh, d, r_cap=self.r_cap, cap=n, group=G, bits=b,
                                 residual=w.residual, device=device)
        c = self.cache
        kt, kh = pinned_u16((bh, n, d))
        vt, vh = pinned_u16((bh, n, d))
        for l in range(L):
            W.fill(w, l, "k", kh)
            W.fill(w, l, "v", vh)
            kd, vd = kt.to(device), vt.to(device)
            K.kivi_quantize_keys(kd, G, b, c.k_codes[l], c.k_scale[l], c.k_zero[l])
            K.kivi_quantize_values(vd, G, b, c.v_codes[l], c.v_scale[l], c.v_zero[l])
            c.k_res[l].copy_(torch.from_numpy(
                W.generate(w, l, "k", tok0=n, n_tok=self.r_cap).view(np.int16)).view(
                    torch.float16).to(device))
            c.v_res[l].copy_(torch.from_numpy(
                W.generate(w, l, "v", tok0=n, n_tok=self.r_cap).view(np.int16)).view(
                    torch.float16).to(device))
        torch.cuda.synchronize(device)
        c.reset(s_q=n, res_head=0, n_res=self.r_cap)
        rng = np.random.default_rng(w.seed)
        self.q_host = torch.from_numpy(
            rng.standard_normal((L, w.batch, self.H_Q, d)).astype(np.float16)).pin_memory()
        self.q = self.q_host.to(device)
        self.out = torch.empty((L, w.batch, self.H_Q, d), dtype=torch.float32, device=device)
        self.scale = 1.0 / d ** 0.5
        self.n_split = K.kivi_decode_attention_splits(c.state, L, w.batch)
        need = K.kivi_decode_attention_workspace(c.state, L, w.batch, self.H_Q, self.n_split)
        self.ws = torch.empty(max(need, 1), dtype=torch.float32, device=device)
        self.q_ptrs = K._ptr_array(list(self.q.unbind(0)), L)
        self.o_ptrs = K._ptr_array(list(self.out.unbind(0)), L)
        per_tok = d * b / 8 * 2 + 8 * d / G * 2          # key + value codes, scales, zeros
        self.tokens = n + self.r_cap
        elems = L * bh * self.tokens * d * 2              # K and V elements attended
        self.kernel_bytes = {"decode_attention": L * bh * (n * per_tok + self.r_cap * d * 4)
                             + self.q.numel() * 2 + self.out.numel() * 4}
        self.step_bytes = self.kernel_bytes["decode_attention"]
        self.step_elems = elems
        self.launches_per_step = 1 if self.n_split == 1 else 2

    def config(self):
        w = self.w
        return {"workload": w.name + "+attention", "layers": w.layers, "batch": w.batch,
                "kv_heads": w.kv_heads, "q_heads": self.H_Q, "head_dim": w.head_dim,
                "bits": w.bits, "group": w.group, "store_tokens": w.store_prefill,
                "residual_tokens": self.r_cap, "n_split": self.n_split,
                "step": "decode attention of one query token per sequence over the packed "
                        "store + fp16 residual of every layer",
                "bytes": "packed codes + scales/zeros + fp16 residual + queries + outputs",
                "fp16_equivalent_bytes_per_step": self.step_elems * 2}

    def step(self, stream, ev=None):
        c = self.cache
        if ev is not None:
            ev[0].record(stream)
        self.K.kivi_decode_attention(c.layers, c.n_layers, c.state, self.w.batch, self.H_Q,
                                     self.scale, self.q_ptrs, self.o_ptrs, self.n_split,
                                     self.ws, stream)
        if ev is not None:
            ev[1].record(stream)

    def step_events(self, evs):
        return evs

    def kernel_times(self, e):
        return {"decode_attention": e[0].elapsed_time(e[1])}

    def e2e_setup(self):
        import torch
        self.out_back = torch.empty(self.out.shape, dtype=torch.float32, pin_memory=True)
        return self.q_host.numel() * 2, self.out_back.numel() * 4

    def e2e_step(self, stream):
        self.q.copy_(self.q_host, non_blocking=True)
        self.step(stream)
        self.out_back.copy_(self.out, non_blocking=True)

    def cpu_sample(self, budget_s: float):
        """The oracle's attention (binary64) over (layer, sequence) pairs of the
        same cache until the budget is spent."""
        import numpy as np
        import oracle as O
        import workloads as W
        w, n = self.w, self.w.store_prefill
        h_kv = w.kv_heads
        done, t_total, pairs = 0.0, 0.0, 0
        q = self.q_host.numpy()
        per_pair = self.step_bytes / (w.layers * w.batch)
        for l in range(w.layers):
            for b in range(w.batch):
                sl = dict(bh0=b * h_kv, bh=h_kv)
                k_st = W.generate(w, l, "k", n_tok=n, **sl)
                v_st = W.generate(w, l, "v", n_tok=n, **sl)
                k_r = W.generate(w, l, "k", tok0=n, n_tok=self.r_cap, **sl)
                v_r = W.generate(w, l, "v", tok0=n, n_tok=self.r_cap, **sl)
                t0 = time.perf_counter()
                kc, ks, kz = O.quantize_keys(k_st, w.group, w.bits)
                vc, vs, vz = O.quantize_values(v_st, w.group, w.bits)
                k = np.concatenate([O.dequantize_keys(kc, ks, kz, n, w.group, w.bits), k_r], 1)
                v = np.concatenate([O.dequantize_values(vc, vs, vz, w.group, w.bits), v_r], 1)
                O.decode_attention(q[l, b:b + 1].view(np.uint16), k, v, self.scale)
                t_total += time.perf_counter() - t0
                done += per_pair
                pairs += 1
                if t_total >= budget_s:
                    return done, t_total, (f"{pairs} (layer, sequence) pairs: quantize, dequantize "
                                           "and binary64 attention of 32 query heads")
        return done, t_total, f"{pairs} (layer, sequence) pairs"


def sweep_inputs(w, device):
    """Keys and values of the store sweep: ((pinned tensor, uint16 view,
    device tensor) for keys, the same for values)."""
    import workloads as W
    out = []
    for kind in ("k", "v"):
        t, h = pinned_u16((w.bh, w.seq, w.head_dim))
        W.fill(w, 0, kind, h)
        out.append((t, h, t.to(device)))
    return tuple(out)


class StoreSweep:
    """Full-tensor quantize of keys and values, then full dequantize, of a
    [bh, S, d] store at one (bits, group) point of the sweep."""

    kernels = ("key_quant", "value_quant", "key_dequant", "value_dequant")
    events_per_step = 5

    def __init__(self, w, device, bits, group, inputs=None):
        import torch
        import kv_cache_quantization_kivi_gb300 as K
        import workloads as W
        self.w, self.K, self.bits, self.group = w, K, bits, group
        bh, S, d = w.bh, w.seq, w.head_dim
        if inputs is None:
            inputs = sweep_inputs(w, device)
        # the store's keys and values do not depend on (bits, G): every cell of
        # the sweep shares one pinned host copy and one device copy
        (self.k_host_t, self.k_host, self.k), (self.v_host_t, self.v_host, self.v) = inputs
        self.kc, self.ks, self.kz = K.kivi_quantize_keys(self.k, group, bits)
        self.vc, self.vs, self.vz = K.kivi_quantize_values(self.v, group, bits)
        self.ky = torch.empty_like(self.k)
        self.vy = torch.empty_like(self.v)
        elems = bh * S * d
        bpe = bytes_per_elem(bits, group)
        self.kernel_bytes = {k: elems * bpe for k in self.kernels}
        self.step_bytes = 4 * elems * bpe
        self.step_elems = 2 * elems
        self.launches_per_step = 4

    def config(self):
        w = self.w
        return {"workload": w.name, "bh": w.bh, "seq": w.seq, "head_dim": w.head_dim,
                "bits": self.bits, "group": self.group,
                "step": "full quantize of keys and values, then full dequantize"}

    def step(self, stream, ev=None):
        K, S, g, b = self.K, self.w.seq, self.group, self.bits
        if ev is not None:
            ev[0].record(stream)
        K.kivi_quantize_keys(self.k, g, b, self.kc, self.ks, self.kz, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        K.kivi_quantize_values(self.v, g, b, self.vc, self.vs, self.vz, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        K.kivi_dequantize_keys(self.kc, self.ks, self.kz, S, g, b, self.ky, stream=stream)
        if ev is not None:
            ev[3].record(stream)
        K.kivi_dequantize_values(self.vc, self.vs, self.vz, g, b, y=self.vy, stream=stream)
        if ev is not None:
            ev[4].record(stream)

    def step_events(self, evs):
        return evs

    def kernel_times(self, e):
        return {"key_quant": e[0].elapsed_time(e[1]), "value_quant": e[1].elapsed_time(e[2]),
                "key_dequant": e[2].elapsed_time(e[3]), "value_dequant": e[3].elapsed_time(e[4])}

    def e2e_setup(self):
        import torch
        self.back = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                     for t in (self.ky, self.vy, self.kc, self.ks, self.kz, self.vc, self.vs,
                               self.vz)]
        h2d = 2 * self.k_host_t.numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in self.back)
        return h2d, d2h

    def e2e_step(self, stream):
        self.k.copy_(self.k_host_t, non_blocking=True)
        self.v.copy_(self.v_host_t, non_blocking=True)
        self.step(stream)
        for dst, src in zip(self.back, (self.ky, self.vy, self.kc, self.ks, self.kz, self.vc,
                                        self.vs, self.vz)):
            dst.copy_(src, non_blocking=True)

    def cpu_sample(self, budget_s: float):
        import oracle as O
        w, g, b = self.w, self.group, self.bits
        done, t_total, rows = 0.0, 0.0, 0
        for i in range(w.bh):
            k = self.k_host[i:i + 1]
            v = self.v_host[i:i + 1]
            t0 = time.perf_counter()
            c, s, z = O.quantize_keys(k, g, b)
            O.dequantize_keys(c, s, z, w.seq, g, b)
            c, s, z = O.quantize_values(v, g, b)
            O.dequantize_values(c, s, z, g, b)
            t_total += time.perf_counter() - t0
            done += 4 * w.seq * w.head_dim * bytes_per_elem(b, g)
            rows += 1
            if t_total >= budget_s:
                break
        return done, t_total, f"{rows} of {w.bh} bh slices (quantize + dequantize, keys and values)"


class FusedStoreSweep(StoreSweep):
    """Full-tensor fused fake quantization of keys and values (codes, scales,
    zeros and the fp16 reconstruction in one pass each) at one sweep point."""

    kernels = ("key_fakequant", "value_fakequant")
    events_per_step = 3

    def __init__(self, w, device, bits, group, inputs=None):
        super().__init__(w, device, bits, group, inputs)
        elems = w.bh * w.seq * w.head_dim
        bpe = fused_bytes_per_elem(bits, group)
        self.kernel_bytes = {k: elems * bpe for k in self.kernels}
        self.step_bytes = 2 * elems * bpe
        self.launches_per_step = 2

    def config(self):
        c = super().config()
        c["step"] = "fused fake quantization of keys and values (store + fp16 reconstruction)"
        c["bytes_per_elem"] = fused_bytes_per_elem(self.bits, self.group)
        return c

    def step(self, stream, ev=None):
        K, g, b = self.K, self.group, self.bits
        if ev is not None:
            ev[0].record(stream)
        K.kivi_fakequant_keys(self.k, g, b, self.ky, True, self.kc, self.ks, self.kz,
                              stream=stream)
        if ev is not None:
            ev[1].record(stream)
        K.kivi_fakequant_values(self.v, g, b, self.vy, True, self.vc, self.vs, self.vz,
                                stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def kernel_times(self, e):
        return {"key_fakequant": e[0].elapsed_time(e[1]),
                "value_fakequant": e[1].elapsed_time(e[2])}

    def cpu_sample(self, budget_s: float):
        done, t, what = super().cpu_sample(budget_s)
        # same oracle work (quantize + dequantize), counted in the fused pass's bytes
        return (done * fused_bytes_per_elem(self.bits, self.group) /
                (2 * bytes_per_elem(self.bits, self.group)), t, what)


def C_void_p_array(evs):
    """ctypes array of the cudaEvent_t handles of torch events (each recorded once)."""
    import ctypes as C
    return (C.c_void_p * len(evs))(*[e.cuda_event for e in evs])


def make_workload(name, device, layers=None, bits=None, group=None, fused=False,
                  attention=False, sink=False):
    import dataclasses
    import workloads as W
    w = W.CONFIGS[name]
    if layers:
        w = dataclasses.replace(w, layers=int(layers))
    if name in ("llama3_2_3b_prefill", "qwen2_5_7b_long", "tiny_flush"):
        if sink:
            return SinkPrefillFlush(w, device)
        return FusedPrefillFlush(w, device) if fused else PrefillFlush(w, device)
    if name == "batched_decode":
        if attention:
            return DecodeAttention(w, device)
        return FusedDecodeFlush(w, device) if fused else DecodeFlush(w, device)
    if name == "large_store_sweep":
        return (FusedStoreSweep if fused else StoreSweep)(w, device, bits or 2, group or 32)
    raise SystemExit(f"unknown workload {name!r}")


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def csrc_hash(kind: str = "flush") -> str:
    """First 16 hex digits of the sha256 of the kernel sources of `kind`."""
    h = hashlib.sha256()
    for f in CSRC_FILES[kind]:
        with open(os.path.join(ROOT, "kv_cache_quantization_kivi_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    wl = d.get("workloads", {}).get(workload, {})
    kind = "attention" if "+attention" in workload else "sink" if "+sink" in workload else "flush"
    if wl.get("csrc_hash") != csrc_hash(kind):
        return None
    entry = wl.get(kernel)
    return None if entry is None else float(entry.get("dram_bytes_per_launch"))


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def time_steps(wl, steps: int, warmup: int, stream, device, sampler=None):
    """W untimed warm-up steps, then exactly K steps between a barrier and a
    synchronize on both sides, with CUDA events on the launching stream
    around the whole region only (an event recorded between two launches
    would end the overlap of a launch with its predecessor's tail); then K
    more steps, outside the timed region, with events around every kernel of
    every step for the per-kernel breakdown.  Returns (elapsed ms of the
    timed K steps, max over ranks; the per-step event lists)."""
    import torch

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    for _ in range(warmup):
        wl.step(stream)
    torch.cuda.synchronize(device)
    start, end = new_events(2)
    torch.cuda.synchronize(device)
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)  # let the sampler start before the load
    barrier()
    torch.cuda.synchronize(device)
    start.record(stream)
    for _ in range(steps):
        wl.step(stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    elapsed = reduce_max(start.elapsed_time(end), device)
    evs = [new_events(wl.events_per_step) for _ in range(steps)]
    handles = [wl.step_events(e) for e in evs]
    torch.cuda.synchronize(device)
    for i in range(steps):
        wl.step(stream, handles[i])
    torch.cuda.synchronize(device)
    return elapsed, evs


def kernel_stats(wl, evs, peak: float) -> dict:
    """Per kernel: average event time, algorithmic GB/s, fraction of the
    measured copy peak and of the nominal 8 TB/s, share of the step's kernel
    time and the spread of the per-step times."""
    k_ms = {k: [] for k in wl.kernels}
    for e in evs:
        for k, t in wl.kernel_times(e).items():
            k_ms[k].append(t)
    total_kernel_ms = sum(sum(v) for v in k_ms.values())
    out = {}
    for k in wl.kernels:
        avg = sum(k_ms[k]) / len(k_ms[k])
        gbs = wl.kernel_bytes[k] / (avg * 1e-3) / 1e9
        out[k] = {"avg_us": round(avg * 1e3, 2), "gbs": round(gbs, 1),
                  "frac_of_measured": round(gbs / peak, 4),
                  "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                  "share": round(sum(k_ms[k]) / total_kernel_ms, 4),
                  **spread_us(k_ms[k])}
    return out


def run_sweep(args, device, stream, peak: float) -> dict:
    """Every (bits, G) cell of the large store sweep, timed like the main
    workload (W warm-up steps, K timed steps, CUDA events per kernel), with
    the SM clocks sampled over the whole sweep."""
    import torch
    import workloads as W
    w = W.CONFIGS["large_store_sweep"]
    inputs = sweep_inputs(w, device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.3)
    cells = {}
    floor = None
    for bits in w.sweep_bits:
        for group in w.sweep_groups:
            cell = (FusedStoreSweep if args.fused else StoreSweep)(w, device, bits, group, inputs)
            ms, evs = time_steps(cell, args.steps, args.warmup, stream, device)
            ks = kernel_stats(cell, evs, peak)
            step_gbs = cell.step_bytes * args.steps / (ms * 1e-3) / 1e9
            cells[f"b{bits}_g{group}"] = {
                "step_gbs": round(step_gbs, 1),
                "ms_per_step": round(ms / args.steps, 5),
                "kernels": {k: {"gbs": v["gbs"], "avg_us": v["avg_us"],
                                "frac_of_measured": v["frac_of_measured"],
                                "frac_of_nominal": v["frac_of_nominal"]}
                            for k, v in ks.items()}}
            lo = min(v["frac_of_nominal"] for v in ks.values())
            floor = lo if floor is None else min(floor, lo)
            del cell
            torch.cuda.synchronize(device)
    clocks = sampler.stop() if not args.no_clocks else None
    kinds = sorted(next(iter(cells.values()))["kernels"])
    at_bar = sum(1 for c in cells.values() for k in c["kernels"].values()
                 if k["frac_of_nominal"] >= 0.70)
    return {"workload": w.name, "bh": w.bh, "seq": w.seq, "head_dim": w.head_dim,
            "step": ("fused fake quantization of keys and values" if args.fused else
                     "full quantize of keys and values, then full dequantize"),
            "cells": cells, "kernels_per_cell": kinds,
            "min_kernel_frac_of_nominal": floor,
            "kernel_cells_at_70pct_of_nominal": f"{at_bar} of {len(cells) * len(kinds)}",
            "clocks": clocks,
            "l2": "no flush: each kernel pass reads and writes 0.6-0.9 GB, more than the "
                  "129 MB L2"}


def run_kivi(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        init_dist("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    import kv_cache_quantization_kivi_gb300 as K
    K.lib()
    wl = make_workload(args.workload, device, args.layers, args.bits, args.group, args.fused,
                       args.attention, args.sink)
    stream = torch.cuda.current_stream(device)
    peak, peak_kind = measured_peaks()

    sampler = ClockSampler(device.index if device.index is not None else 0)
    elapsed_ms, evs = time_steps(wl, args.steps, args.warmup, stream, device,
                                 None if args.no_clocks else sampler)
    clocks = sampler.stop() if not args.no_clocks else None
    ms_per_step = elapsed_ms / args.steps
    total_bytes = reduce_sum(wl.step_bytes * args.steps, device)
    value = total_bytes / (elapsed_ms * 1e-3) / 1e9

    kernels = kernel_stats(wl, evs, peak)
    k_total = {k: v["avg_us"] for k, v in kernels.items()}
    dom = max(wl.kernels, key=lambda k: k_total[k])
    dom_avg_s = kernels[dom]["avg_us"] * 1e-6
    achieved = wl.kernel_bytes[dom] / dom_avg_s / 1e9
    traffic = ncu_traffic(args.workload + ("+fused" if args.fused else "")
                          + ("+attention" if args.attention else "")
                          + ("+sink" if args.sink else ""), dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "algorithmic_bytes_per_launch": wl.kernel_bytes[dom], "traffic": traffic}

    # end to end: pinned host inputs -> device -> kernels -> host
    e2e = None
    if args.e2e_steps > 0:
        h2d, d2h = wl.e2e_setup()
        wl.e2e_step(stream)
        torch.cuda.synchronize(device)
        a, b = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        barrier()
        torch.cuda.synchronize(device)
        a.record(stream)
        for _ in range(args.e2e_steps):
            wl.e2e_step(stream)
        b.record(stream)
        torch.cuda.synchronize(device)
        e_ms = reduce_max(a.elapsed_time(b), device)
        e_bytes = reduce_sum(wl.step_bytes * args.e2e_steps, device)
        e2e = {"value": round(e_bytes / (e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
               "ms_per_step": round(e_ms / args.e2e_steps, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        if getattr(wl, "e2e_pipeline", None):
            e2e["pipeline"] = wl.e2e_pipeline

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cb, cs, what = wl.cpu_sample(args.cpu_seconds)
        cpu = {"value": round(cb / cs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{what}; {cs:.1f} s single-threaded on the host", **host_cpu()}

    # what the line reports about the main workload, taken before its buffers
    # are released for the sweep
    config = wl.config()
    config["bytes_per_step"] = wl.step_bytes
    config["fp16_elements_per_step"] = wl.step_elems
    config["l2"] = ("no flush: each step reads and writes ~%.2f GB, more than the 129 MB L2"
                    % (wl.step_bytes / 1e9))
    config["parallelism"] = f"independent replicas x{ws}" if ws > 1 else "single GPU"
    launches = wl.launches_per_step * args.steps
    elems = reduce_sum(wl.step_elems * args.steps, device)

    sweep = None
    if not args.no_sweep and args.workload == DEFAULT_WORKLOAD and not args.attention \
            and not args.sink:
        del wl
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
        sweep = run_sweep(args, device, stream, peak)
        launches += sum(len(c["kernels"]) for c in sweep["cells"].values()) * args.steps

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "formats": {"inputs_and_reconstructions": "fp16", "codes": "u32 (packed)",
                    "scale_zero": "f32"},
        "data": "synthetic (seeded counter-based generator, shapes of the pages' models)",
        "config": config,
        "pct_of_hbm_peak": {"measured_copy": round(value / ws / peak * 100, 2),
                            "nominal_8tbs": round(value / ws / NOMINAL_HBM_GBS * 100, 2)},
        "elements_per_s": round(elems / (elapsed_ms * 1e-3), 1),
        "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "sweep": sweep, "gpu_launches": launches, "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.json_out and rank == 0:
        with open(args.json_out, "w") as f:
            json.dump(line, f, indent=1)


def run_reference(args):
    """The CPU oracle, as it stands, on the same metric and workload: each step
    is a bounded sample (a slice of one layer's flush + dequantize) sized so
    that warmup + steps end within a few minutes."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle as O
    import workloads as W
    w = W.CONFIGS[args.workload]
    O.lib()
    n = O.flush_size(w.seq, w.residual, w.group)
    budget = args.reference_seconds
    per_step = budget / max(1, args.steps + args.warmup)
    # ~26 ns per element-operation measured for this oracle; 4 operations per element
    est_ns_per_token_bh = 4 * w.head_dim * 30e-9
    bh_tokens = max(w.group, int(per_step / est_ns_per_token_bh) // w.group * w.group)
    tokens = min(n, bh_tokens)
    bh = max(1, min(w.bh, bh_tokens // max(tokens, 1)))
    tok_res = tokens + w.residual if tokens + w.residual <= w.seq else w.seq
    tok_res = -(-tok_res // w.group) * w.group
    samples = []
    for l in range(min(w.layers, 4)):
        k = np.ascontiguousarray(W.generate(w, l, "k", n_tok=tok_res, bh=bh))
        v = np.ascontiguousarray(W.generate(w, l, "v", n_tok=tok_res, bh=bh))
        samples.append((k, v))
    Wd = 32 // w.bits

    def one(i):
        k, v = samples[i % len(samples)]
        st = O.Store(bh, w.head_dim, tok_res, w.group, w.bits)
        m, _, _, _ = O.flush(k, v, st, w.residual, 0, 0, tok_res)
        O.dequantize_keys(st.k_codes[:, :m // Wd], st.k_scale[:, :m // w.group],
                          st.k_zero[:, :m // w.group], m, w.group, w.bits)
        O.dequantize_values(st.v_codes[:, :m], st.v_scale[:, :m], st.v_zero[:, :m],
                            w.group, w.bits)
        return 4 * bh * m * w.head_dim * bytes_per_elem(w.bits, w.group)

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    total = 0.0
    for i in range(args.steps):
        total += one(i)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    sample = (f"each step: {bh} of {w.bh} bh x {tok_res} tokens of one layer "
              f"(flush of {tok_res - w.residual if tok_res - w.residual > 0 else 0} tokens + "
              f"dequantize, keys and values); single-threaded")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.layers, "bh": w.bh, "seq": w.seq,
                       "head_dim": w.head_dim, "bits": w.bits, "group": w.group,
                       "residual": w.residual},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample, **host_cpu()},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def relaunch_distributed(n: int, argv) -> int:
    """Runs this script under torch.distributed.run with one process per GPU
    (rendezvous on 127.0.0.1); returns its exit status."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=None,
                    help="GPUs (processes, one per GPU); default: WORLD_SIZE under torchrun, "
                         "else 1")
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("kivi", "reference"), default="kivi")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="time budget of the oracle CPU-baseline sample")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="total oracle time budget of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave out the nine (bits, G) cells of the large store sweep that "
                         "follow the default workload in the same line")
    ap.add_argument("--json-out", default=None)
    ap.add_argument("--bits", type=int, default=None, help="large_store_sweep: code width")
    ap.add_argument("--group", type=int, default=None, help="large_store_sweep: group size")
    ap.add_argument("--fused", action="store_true",
                    help="time the fused fake-quant form (store and fp16 reconstruction in "
                         "one pass) instead of quantize + dequantize")
    ap.add_argument("--sink", action="store_true",
                    help="prefill workloads: the KIVI-Sink flush (scores, top-5, protected "
                         "flush, dequantize, restore)")
    ap.add_argument("--attention", action="store_true",
                    help="batched_decode: time decode attention over the packed cache")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (profiling runs only; "
                         "the reported config says so)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws = int(os.environ.get("WORLD_SIZE", "0"))
    if args.gpus is None:
        args.gpus = ws or 1
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if ws == 0 and args.gpus > 1:
        # not under torchrun yet: one process per GPU, launched the same way
        sys.exit(relaunch_distributed(args.gpus, sys.argv[1:] if argv is None else argv))
    if ws not in (0, args.gpus):
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {ws}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kivi(args)


if __name__ == "__main__":
    main()
