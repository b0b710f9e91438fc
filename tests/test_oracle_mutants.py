"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of ``oracle/kivi_oracle.c`` (in a
temporary directory; the repository's file is never touched), builds it
with the oracle's own flags, and runs the pin file that should catch it
against that build (``KIVI_ORACLE_LIB``).  The pins must fail.  The
mistakes: the rounding rule, a fused reconstruction, zero padding, a sign,
signed-zero handling, bit order, the level count, the flush size, a
reciprocal for the division, truncating fp16 conversion, a group index,
the ring row and the count of an append;
for KIVI-Sink the calibration exclusion, a sink's code, the tie rule, the
mean over heads, the square root, the restore row, the value row and the
store capacity; for attention the maximum subtraction, the scale, the key
and value indexing, the normalisation, the query head and the maximum
itself.  (Writing the value packing with the token index in place of the
channel index is not among them: in that function the two coincide, an
equivalent rewrite.)
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kivi_oracle.c")
HDR = os.path.join(ROOT, "oracle", "kivi_oracle.h")

PINS = "tests/test_oracle_pins.py"
SINK = "tests/test_oracle_sink_pins.py"
ATTN = "tests/test_oracle_attention_pins.py"

MUTANTS = {
    # flush path
    "half_away_from_zero": (PINS, "float r = nearbyintf(u);", "float r = roundf(u);"),
    "fused_reconstruction": (PINS, "volatile float prod = (float)q * scale;\n    const float r = prod + zero;",
                             "const float r = fmaf((float)q, scale, zero);"),
    "zero_padding": (PINS, "    if (t > s - 1) t = s - 1;\n    return kivi_oracle_half_to_float(x_bh[t * d + c]);",
                     "    if (t > s - 1) return 0.0f;\n    return kivi_oracle_half_to_float(x_bh[t * d + c]);"),
    "sign": (PINS, "const float t = x - zero;", "const float t = zero - x;"),
    "no_zero_canonicalisation": (PINS, "    mn = mn + 0.0f;\n    mx = mx + 0.0f;", ""),
    "msb_first_keys": (PINS, "words[i / w] |= q[i] << ((i % w) * bits);",
                       "words[i / w] |= q[i] << ((w - 1 - i % w) * bits);"),
    "levels_2_pow_b": (PINS, "*scale = (mx - mn) / (float)qmax_of(bits);",
                       "*scale = (mx - mn) / (float)(1u << bits);"),
    "flush_size_rounds_up": (PINS, "return ((n_res - residual) / group) * group;",
                             "return ((n_res - residual + group - 1) / group) * group;"),
    "reciprocal": (PINS, "const float u = t / scale;", "const float u = t * (1.0f / scale);"),
    "truncating_fp16": (PINS, "float n = nearbyintf(units);", "float n = truncf(units);"),
    "append_row": (PINS, "const int64_t row = (res_head + *n_res + i) % r_cap;",
                   "const int64_t row = (res_head + i) % r_cap;"),
    "append_count": (PINS, "    *n_res += n;\n    return 0;", "    return 0;"),
    "key_dequant_group_index": (PINS, "const int64_t p = (b * ng + t / group) * d + c;",
                                "const int64_t p = (b * ng + t / w / group) * d + c;"),
    # KIVI-Sink
    "sink_not_excluded": (SINK, "                    if (is_sink(top, top_count[b], *s_q + li)) continue;\n", ""),
    "sink_code": (SINK, "for (int i = 0; i < group; ++i) q[i] = 0u;            /* sink tokens: code 0 */",
                  "for (int i = 0; i < group; ++i) q[i] = 1u;"),
    "tie_to_later": (SINK, "return sa > sb || (sa == sb && pa < pb);",
                     "return sa > sb || (sa == sb && pa > pb);"),
    "no_mean_over_heads": (SINK, "score[b * n + t] = sum / (float)heads;", "score[b * n + t] = sum;"),
    "no_sqrt": (SINK, "sum = sum + sqrtf(acc);", "sum = sum + acc;"),
    "restore_row": (SINK, "memcpy(k + (bb * s + t) * d, sink_k + (bb * sink_cap + j) * d,",
                    "memcpy(k + (bb * s + (t > 0 ? t - 1 : t)) * d, sink_k + (bb * sink_cap + j) * d,"),
    "sink_value_row_quantized": (
        SINK,
        "                for (int64_t g2 = 0; g2 < d / group; ++g2) { vs[g2] = 0.0f; vz[g2] = 0.0f; }\n"
        "                continue;",
        "                for (int64_t g2 = 0; g2 < d / group; ++g2) { vs[g2] = 0.0f; vz[g2] = 0.0f; }"),
    "no_capacity_check": (SINK, "if (sink_count[b] + add > sink_cap) return -3;", "(void)add;"),
    # attention
    "no_max_subtraction": (ATTN, "s[t] = exp(s[t] - mx);", "s[t] = exp(s[t]);"),
    "no_scale": (ATTN, "s[t] = scale * dot;", "s[t] = dot;"),
    "key_index": (ATTN, "(double)kivi_oracle_half_to_float(k[t * d + c]);",
                  "(double)kivi_oracle_half_to_float(k[c * n + t < n * d ? c * n + t : 0]);"),
    "no_normalisation": (ATTN, "acc += (s[t] / den) *", "acc += s[t] *"),
    "query_head": (ATTN, "(double)kivi_oracle_half_to_float(q[h * d + c]) *",
                   "(double)kivi_oracle_half_to_float(q[c]) *"),
    "value_index": (ATTN, "(double)kivi_oracle_half_to_float(v[t * d + c]);",
                    "(double)kivi_oracle_half_to_float(v[t * d + (d - 1 - c)]);"),
    "wrong_maximum": (ATTN, "if (s[t] > mx) mx = s[t];", "if (s[t] < mx || mx == -INFINITY) mx = s[t];"),
}


@pytest.fixture(scope="module")
def cc():
    c = os.environ.get("CC", "gcc")
    if shutil.which(c) is None:
        pytest.skip("no C compiler")
    return c


def _build_copy(cc, tmp_path, text):
    shutil.copy(HDR, tmp_path / "kivi_oracle.h")
    (tmp_path / "kivi_oracle.c").write_text(text)
    lib = tmp_path / "libkivi_oracle_copy.so"
    subprocess.run([cc, *oracle.CFLAGS, str(tmp_path / "kivi_oracle.c"), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    return lib


def _run_pins(lib, *files):
    env = dict(os.environ, KIVI_ORACLE_LIB=str(lib))
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-m", "not gpu", *files], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_unchanged_copy_passes_every_pin(cc, tmp_path):
    """Control: the unmodified source, built and loaded the same way, passes."""
    r = _run_pins(_build_copy(cc, tmp_path, open(SRC).read()), PINS, SINK, ATTN)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, cc, tmp_path):
    pins, find, replace = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(find) == 1, f"{name}: the planted site is no longer in the oracle"
    r = _run_pins(_build_copy(cc, tmp_path, src.replace(find, replace)), pins)
    # exit code 1: a pin failed; a negative code: the run died of a signal (the
    # mutant without the sink store's capacity check writes past the store).
    # A collection error (2-4) or no tests (5) would not count.
    assert r.returncode == 1 or r.returncode < 0, \
        f"{name}: pins did not catch it (exit {r.returncode})\n{r.stdout[-2000:]}"
