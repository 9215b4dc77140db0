"""Build the sm_103a shared library ``libra_gb300.so`` in this directory.

Every CUDA source is compiled for sm_103a only (``-gencode
arch=compute_103a,code=sm_103a``), host sources with the same nvcc driver;
translation units compile in parallel and link into one shared object with
the static CUDA runtime, so the library depends on no CUDA shared object at
load time (the CUDA driver API is looked up through the runtime when first needed).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libra_gb300.so")

SOURCES = ["ra_api.cpp", "ra_sched.cpp", "ra_misc.cu", "attn_f32.cu", "attn_tc_sm103.cu",
           "decode_attn.cu", "ra_noalloc.cu", "ra_selftest.cu", "ra_tma.cpp",
           "decode_tc_sm103.cu", "attn_pair_sm103.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build")
    return cand


def _compile(nvcc, src, extra):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc, "-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
           "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cu"):
        cmd += ARCH + ["-lineinfo", "--expt-relaxed-constexpr"] + extra
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(verbose=False, ptxas_info=False):
    """Compile and link; returns the library path.  Raises on any error."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs = []
    logs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, rc, out in ex.map(lambda s: _compile(nvcc, s, extra), SOURCES):
            logs.append((src, out))
            if rc != 0:
                raise RuntimeError(f"compiling {src} failed:\n{out}")
            objs.append(obj)
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-cudart", "static", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        for src, out in logs:
            if out.strip():
                print(f"--- {src}\n{out}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
