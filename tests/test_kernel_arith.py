"""Host checks of arithmetic the CUDA kernels rely on for bit-exactness.

The quantize kernels compute the group scale RN((max - min) / Q), Q = 2^b - 1,
without a division: q0 = RN(x * RN(1/Q)), one fused multiply-add for the exact
residual and one for the correction (tests/native/divq_check.c).  It must equal
the IEEE quotient for every finite x >= 0; the full check (stride 1, all 2^31
patterns, about a minute on 8 cores) passed; this test runs it on every 61st
bit pattern, which still covers every exponent and the whole mantissa range.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def divq(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("divq") / "divq_check")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                    os.path.join(HERE, "native", "divq_check.c"), "-o", exe, "-lm"], check=True)
    return exe


def test_division_by_q_equals_ieee_quotient(divq):
    r = subprocess.run([divq, "61"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 3 and all("mismatches=0" in l for l in lines), r.stdout
    assert all(int(l.split("checked=")[1].split()[0]) > 30_000_000 for l in lines)
