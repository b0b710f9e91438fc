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


def _byte_perm(x: int, y: int, s: int) -> int:
    """CUDA __byte_perm in its default mode: byte n of the result is byte
    (nibble n of s) of the eight bytes y:x (x bytes 0-3, y bytes 4-7); the
    nibbles here stay below 8, so no sign replication applies."""
    src = (y << 32) | x
    out = 0
    for n in range(4):
        sel = (s >> (4 * n)) & 0xF
        assert sel < 8
        out |= ((src >> (8 * sel)) & 0xFF) << (8 * n)
    return out


def test_two_bit_value_table_lookup_selects_each_code():
    """The 2-bit value dequantizer looks its fp16 values up in an 8-byte table
    (code q at bytes 2q, 2q + 1: codes 0, 1 in the low register, 2, 3 in the
    high one) with byte permutes whose selectors it builds from one byte of
    four codes: spread one code to a byte, then q * 0x22 + 0x10 per byte.
    For every code byte, both selectors fetch exactly the four codes' table
    entries, in channel order."""
    vals = [0x1234, 0xABCD, 0x5A5A, 0xF00F]               # distinct 16-bit entries
    lo = vals[0] | (vals[1] << 16)
    hi = vals[2] | (vals[3] << 16)
    for b in range(256):
        q = [(b >> (2 * j)) & 3 for j in range(4)]
        x = (b | (b << 12)) & 0x000F000F
        x = (x | (x << 6)) & 0x03030303
        assert [(x >> (8 * j)) & 0xFF for j in range(4)] == q
        sel = (x * 0x22 + 0x10101010) & 0xFFFFFFFF
        first = _byte_perm(lo, hi, sel & 0xFFFF)
        second = _byte_perm(lo, hi, sel >> 16)
        assert first == vals[q[0]] | (vals[q[1]] << 16)
        assert second == vals[q[2]] | (vals[q[3]] << 16)
