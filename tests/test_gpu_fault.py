"""The bounded-wait failure path on the GPU, without a fault: a warp waits,
with the decode-attention pipeline's bounded mbarrier wait, on a phase that
nothing completes; the wait gives up after its limit, the device fault word
records it, the host reads and clears it, and the context stays usable."""
from __future__ import annotations

import time

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_same, host_u32, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_cache_quantization_kivi_gb300 as K  # noqa: E402


def test_bounded_wait_gives_up_and_reports():
    torch.cuda.synchronize()
    assert K.kivi_device_fault() == 0
    t0 = time.perf_counter()
    K.kivi_selftest_wait_timeout(50_000)          # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert K.kivi_device_fault() == 4             # bit 2: the self-test's wait gave up
    assert K.kivi_device_fault() == 0             # read and cleared
    assert 0.045 < dt < 5.0
    # the context is still usable: a quantize call matches the oracle
    w = W.custom(seed=3, kv_heads=2, seq=64, head_dim=128)
    x = W.generate(w, 0, "k")
    c, _, _ = K.kivi_quantize_keys(to_dev(x), 32, 2)
    torch.cuda.synchronize()
    assert_same("codes after the timeout", host_u32(c), O.quantize_keys(x, 32, 2)[0])
    assert K.kivi_device_fault() == 0


def test_selftest_limits_are_checked_on_the_host():
    assert K.lib().kivi_selftest_wait_timeout(0, None) == 1
    assert K.lib().kivi_selftest_wait_timeout(1_000_001, None) == 1
    assert np.uint32(K.kivi_device_fault()) == 0
