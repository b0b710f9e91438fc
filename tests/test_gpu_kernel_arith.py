"""GPU checks of the quantize kernels' arithmetic, each compiled against the
kernels' own headers: the group reciprocal (kivi_arith.cuh) is bit-identical
to the correctly rounded reciprocal for every normal float in [2^-126,
2^126), the whole range a group scale can take and more; the per-element
code of both fast paths (kivi_device.cuh: codes2, the fused multiply-add
form with its exact fallback, and codes2_diff_nobranch, difference first,
whose declined pairs the kernels redo exactly) equals the literal definition
with the IEEE division on random binary16 groups and on elements next to a
rounding midpoint."""
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


def build_and_run(tmp_path, name):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / name)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    os.path.join(HERE, "native", name + ".cu"), "-o", exe], check=True)
    return subprocess.run([exe], capture_output=True, text=True, timeout=300)


def test_reciprocal_equals_correctly_rounded_everywhere(tmp_path):
    r = build_and_run(tmp_path, "rcp_check")
    assert r.returncode == 0, r.stdout + r.stderr
    assert "checked=2113929216 mismatches=0" in r.stdout


def test_codes_equal_the_literal_definition(tmp_path):
    r = build_and_run(tmp_path, "quot_check")
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 4 and all("mismatches=0" in l for l in lines), r.stdout
    # the difference-first path declines few random pairs (its bound does not
    # grow with the group's distance from zero)
    rnd = [l for l in lines if "difference-first" in l and "mode=random" in l][0]
    samples = int(rnd.split("samples=")[1].split()[0])
    assert int(rnd.split("declined=")[1]) < samples // 1000, rnd
