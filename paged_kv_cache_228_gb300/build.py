"""Build libpa.so in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_228_gb300.build [--force]

One nvcc invocation per translation unit (the CUDA kernels + C ABI in
``csrc/libpa.cu``; the host block manager in ``csrc/block_manager.cpp``),
run in parallel, then one link.  The CUDA runtime is linked statically; the
driver API is reached at run time through ``cudaGetDriverEntryPointByVersion``
so the library has no link dependency on ``libcuda``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}"]

SOURCES = ["libpa.cu", "block_manager.cpp"]
DEPS = ["libpa.cu", "block_manager.cpp", "decode.cuh", "decode_tc.cuh", "cache_ops.cuh",
        "cascade.cuh", "nvfp4.cuh", "pa_device.cuh", "umma.cuh"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    files = [os.path.join(CSRC, f) for f in DEPS] + [os.path.join(INCLUDE, "pa.h"),
                                                      os.path.join(INCLUDE, "pa_testing.h"),
                                                      os.path.abspath(__file__)]
    return any(os.path.getmtime(f) > t for f in files)


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile libpa.so if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        cmds.append(cmd)
    with ThreadPoolExecutor(len(cmds)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=force or bool(extra), verbose=True, extra=extra))
