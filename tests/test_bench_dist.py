"""bench.py's multi-process path on CPU: world size 2 over gloo.  The data
path has no collective; only the step time (max over ranks) and the byte
count (sum over ranks) are reduced, and only rank 0 prints."""
from __future__ import annotations

import os
import subprocess
import sys
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
ws, rank = bench.init_dist("gloo")
assert ws == 2
mx = bench.reduce_max(10.0 + rank)
sm = bench.reduce_sum(3.0 * (rank + 1))
bench.barrier()
print(f"rank={{rank}} max={{mx}} sum={{sm}}", flush=True)
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _launch(code, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code] if code else [sys.executable, *args]
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True, cwd=ROOT))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=240)
        outs.append((p.returncode, o, e))
    return outs


def test_timing_reductions_over_two_gloo_ranks():
    outs = _launch(CHILD.format(root=ROOT))
    for rc, o, e in outs:
        assert rc == 0, e
        assert "max=11.0" in o and "sum=9.0" in o


def test_reference_arm_prints_on_rank_zero_only():
    outs = _launch(None, args=("bench.py", "--impl", "reference", "--steps", "3",
                               "--warmup", "3", "--reference-seconds", "3"))
    (rc0, o0, e0), (rc1, o1, e1) = outs
    assert rc0 == 0 and rc1 == 0, (e0, e1)
    assert '"impl": "reference"' in o0 and o1.strip() == ""


def test_gpus_flag_must_match_the_launch():
    """--gpus that contradicts torchrun's WORLD_SIZE is an error, not ignored."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "3", "--impl", "reference"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def test_gpus_flag_relaunches_under_torchrun():
    """--gpus 2 outside torchrun starts two ranks (gloo-free: the reference arm
    prints on rank 0 only)."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--reference-seconds", "3"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr
    assert r.stdout.count('"impl": "reference"') == 1
