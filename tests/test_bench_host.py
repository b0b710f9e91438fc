"""Host logic of bench.py that needs no GPU: the layer chunks of the
end-to-end pipeline."""
from __future__ import annotations

import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("layers", [1, 2, 3, 4, 5, 7, 9, 16, 28, 32, 36, 80, 128])
@pytest.mark.parametrize("chunks,ramp", [(5, (1, 1, 2, 2)), (7, (1, 1, 2)), (7, ()), (14, (1, 1))])
def test_e2e_bounds_cover_every_layer_once(layers, chunks, ramp):
    b = load_bench().e2e_bounds(layers, chunks, ramp)
    assert b[0] == 0 and b[-1] == layers
    assert all(x < y for x, y in zip(b, b[1:]))          # non-empty chunks, in order
    sizes = [y - x for x, y in zip(b, b[1:])]
    base = -(-layers // chunks)
    # the ramp's sizes lead, each below the base chunk; no later chunk is
    # far above the base size
    lead = [r for r in ramp if r < base]
    k = 0
    while k < len(lead) and sum(lead[:k + 1]) <= layers:
        k += 1
    assert sizes[:k] == lead[:k]
    assert max(sizes) <= 2 * base


def test_e2e_bounds_of_the_benchmarked_prefill():
    bench = load_bench()
    b = bench.e2e_bounds(28, bench.PrefillFlush.E2E_CHUNKS, bench.PrefillFlush.E2E_RAMP)
    assert b == [0, 1, 2, 4, 8, 12, 16, 20, 24, 28]


def test_kernel_time_spread():
    """Median, extremes and interquartile range of per-step kernel times."""
    bench = load_bench()
    ms = [0.050, 0.051, 0.049, 0.052, 0.050, 0.060, 0.048]   # sorted: 48 49 50 50 51 52 60 us
    s = bench.spread_us(ms)
    assert s["median_us"] == 50.0 and s["min_us"] == 48.0 and s["max_us"] == 60.0
    assert s["iqr_pct"] == 4.0                                 # (51.5 - 49.5) / 50
    assert bench.spread_us([0.1]) == {"median_us": 100.0, "min_us": 100.0, "max_us": 100.0,
                                      "iqr_pct": 0.0}


def test_host_cpu_description():
    info = load_bench().host_cpu()
    assert info["nproc"] >= 1 and isinstance(info["cpu_model"], str) and info["cpu_model"]


def test_decode_config_reports_residual_and_compaction():
    """The decode flush's config keeps the residual length as a number and
    states the compaction bytes (none: the residual is a ring)."""
    bench = load_bench()
    import workloads as W
    d = bench.DecodeFlush.__new__(bench.DecodeFlush)
    d.w, d.cycle = W.CONFIGS["batched_decode"], 100
    c = d.config()
    assert c["residual"] == 32 and c["residual_compaction_bytes_per_step"] == 0
    assert c["workload"] == "batched_decode" and c["tokens_flushed_per_step"] == 32


def test_cpu_sample_times_each_oracle_function():
    """The benchmark's CPU leg (the oracle's flush and both dequantizations of
    whole layers) on the tiny workload: bytes, time and a per-function
    breakdown."""
    import numpy as np
    import oracle as O
    import workloads as W
    bench = load_bench()
    w = W.CONFIGS["tiny_flush"]
    pf = bench.PrefillFlush.__new__(bench.PrefillFlush)
    pf.w = w
    pf.n = O.flush_size(w.seq, w.residual, w.group)
    shape = (w.layers, w.bh, w.seq, w.head_dim)
    pf.k_host = np.zeros(shape, np.uint16)
    pf.v_host = np.zeros(shape, np.uint16)
    for l in range(w.layers):
        W.fill(w, l, "k", pf.k_host[l])
        W.fill(w, l, "v", pf.v_host[l])
    done, secs, what = pf.cpu_sample(0.0)                 # stops after one layer
    elems = w.bh * pf.n * w.head_dim
    assert done == 4 * elems * bench.bytes_per_elem(w.bits, w.group) and secs > 0
    assert what.startswith("1 of 1 layers") and "dequantize_values" in what


def test_every_kernel_source_is_built_and_hashed():
    """Every file under csrc/ is compiled (a translation unit) or tracked as
    a header by the build, and every file the kernels of a workload family
    include is in that family's hash (bench.py CSRC_FILES), so a committed
    ncu traffic figure goes stale whenever a kernel it measured changes."""
    import re
    import kv_cache_quantization_kivi_gb300._build as B
    bench = load_bench()
    csrc = B.CSRC
    files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    assert sorted(B.SOURCES + B.HEADERS) == files
    inc = re.compile(r'#include "([^"/]+)"')

    def closure(names):
        seen, todo = set(), list(names)
        while todo:
            f = todo.pop()
            if f in seen or not os.path.exists(os.path.join(csrc, f)):
                continue
            seen.add(f)
            todo += inc.findall(open(os.path.join(csrc, f)).read())
        return seen

    fams = bench.CSRC_FILES
    for fam, tus in {"flush": ["kivi_keys.cu", "kivi_values.cu", "kivi_staged.cu", "kivi_ring.cu"],
                     "attention": ["kivi_attention.cu", "kivi_attention_d64.cu",
                                   "kivi_attention_d256.cu", "kivi_attention_ws.cu"],
                     "sink": ["kivi_sink.cu", "kivi_keys.cu", "kivi_values.cu",
                              "kivi_staged.cu"]}.items():
        missing = closure(tus) - set(fams[fam])
        assert not missing, (fam, missing)
