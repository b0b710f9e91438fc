"""GPU check of the reciprocal the quantize kernels use for a group's fast
path (kivi_arith.cuh): bit-identical to the correctly rounded reciprocal
for every normal float in [2^-126, 2^126), the whole range a group scale can
take and more.  The checker includes the kernels' own header."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_equals_correctly_rounded_everywhere(tmp_path):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "rcp_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    os.path.join(HERE, "native", "rcp_check.cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "checked=2113929216 mismatches=0" in r.stdout
