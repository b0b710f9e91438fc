"""The benchmark's end-to-end step (pinned host buffers, host-to-device copies,
the C-ABI flush and dequantize over layer chunks on three streams, captured
in a CUDA graph, device-to-host copies) returns exactly what the plain
on-device step computes, and that equals the oracle on sampled groups: the
pipelined copies neither race the kernels nor each other."""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import pytest

import oracle as O
from gpu_util import sample_keys, sample_values

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def bits_of(t):
    return t.cpu().numpy().view(np.uint32) if t.dtype == torch.float32 else \
        t.cpu().numpy().view(np.uint16 if t.dtype == torch.float16 else np.uint32)


@pytest.mark.parametrize("layers", [3, 9])
def test_pipelined_e2e_step_equals_device_step(layers):
    bench = load_bench()
    dev = torch.device("cuda", 0)
    wl = bench.make_workload("llama3_2_3b_prefill", dev, layers)
    stream = torch.cuda.current_stream(dev)
    wl.e2e_setup()
    # poison the host result buffers, then one pipelined step (capture + replay)
    for t in [wl.k_back, wl.v_back] + wl.store_back:
        t.fill_(0)
    wl.e2e_step(stream)
    wl.e2e_step(stream)          # a replay of the captured graph
    torch.cuda.synchronize(dev)
    host = [bits_of(t).copy() for t in [wl.k_back, wl.v_back] + wl.store_back]
    # the plain device step on the same residual windows
    wl.step(stream)
    torch.cuda.synchronize(dev)
    dev_out = [bits_of(t) for t in [wl.k_out, wl.v_out] + wl.store_dev]
    for a, b in zip(host, dev_out):
        assert np.array_equal(a, b)
    # and the oracle on sampled groups of the first and last layer
    w = wl.w
    n = wl.n
    rng = np.random.default_rng(layers)
    kc, ks, kz, vc, vs, vz = host[2:]
    for l in (0, layers - 1):
        k = np.ascontiguousarray(wl.k_host[l][:, :n])
        v = np.ascontiguousarray(wl.v_host[l][:, :n])
        sample_keys(k, kc[l], ks[l], kz[l], host[0][l], w.group, w.bits, 60, rng)
        sample_values(v, vc[l], vs[l], vz[l], host[1][l], w.group, w.bits, 60, rng)
    assert O.flush_size(w.seq, w.residual, w.group) == n
