"""The index-checking build (KIVI_DEBUG_BOUNDS): the small-case parity suites
of the flush and full-tensor paths run once against ``libkivi_debug.so``, in
which every global access of the quantize, dequantize and append kernels
checks its offset against its bh slice and records a failure in bit 4 of the
device fault word instead of touching memory.  Every test must pass with the
bit clear after it (checked by the autouse fixture of conftest.py)."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_fakequant.py", "tests/test_gpu_append.py",
          "tests/test_gpu_flush_shapes.py"]


def test_parity_suites_under_index_checks():
    from kv_cache_quantization_kivi_gb300 import _build
    _build.build(debug_bounds=True)
    env = dict(os.environ, KIVI_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-x", "-m", "gpu",
                        "-k", "not full_size", "-p", "no:cacheprovider"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "libkivi_debug.so" in r.stdout, r.stdout[-2000:]
