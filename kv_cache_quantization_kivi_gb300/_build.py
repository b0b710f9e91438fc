"""Builds the CUDA library ``libkivi.so`` in-tree with nvcc for sm_103a.

The three translation units compile in parallel; the shared object links the
CUDA runtime statically, so the library depends on the driver only.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libkivi.so")
# the index-checking build (KIVI_DEBUG_BOUNDS: every global access of the
# flush and full-tensor kernels checked against its bh slice, failures
# recorded in the device fault word), loaded when KIVI_DEBUG_BOUNDS=1
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libkivi_debug.so")
HEADER = os.path.join(ROOT, "include", "kivi.h")

SOURCES = ["kivi_api.cu", "kivi_keys.cu", "kivi_values.cu", "kivi_attention.cu",
           "kivi_attention_d64.cu", "kivi_attention_d256.cu", "kivi_attention_ws.cu",
           "kivi_sink.cu",
           "kivi_ring.cu", "kivi_staged.cu"]
HEADERS = ["kivi_device.cuh", "kivi_arith.cuh", "kivi_launch.h", "kivi_dispatch.h",
           "kivi_expand.cuh", "kivi_attention_kernel.cuh", "kivi_tc_common.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] +
            [os.path.join(CSRC, h) for h in HEADERS] + [HEADER, os.path.abspath(__file__)])


def is_stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug_bounds: bool = False) -> str:
    """Compile and link ``libkivi.so`` (``libkivi_debug.so`` with
    ``debug_bounds``) if missing or older than its sources."""
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    if not force and not is_stale(lib_path):
        return lib_path
    os.makedirs(OUT_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug_bounds:
        extra.append("-DKIVI_DEBUG_BOUNDS")
    pid = os.getpid()
    tag = "dbg" if debug_bounds else "rel"

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR, f"{os.path.splitext(src)[0]}.{tag}.{pid}.o")
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    objs = [os.path.join(OUT_DIR, f"{os.path.splitext(s)[0]}.{tag}.{pid}.o") for s in SOURCES]
    tmp = lib_path + f".{pid}.tmp"
    try:
        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            list(ex.map(compile_one, SOURCES))
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
    finally:
        for o in objs:
            try:
                os.remove(o)
            except OSError:
                pass
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
