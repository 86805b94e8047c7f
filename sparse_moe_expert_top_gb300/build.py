"""Builds the CUDA library in-tree: csrc/*.cu -> lib/libmoe_gb300.so (sm_103a only).

The translation units are compiled in parallel with nvcc and linked into
one shared library with a static CUDA runtime.  Usage:

    python -m sparse_moe_expert_top_gb300.build [--verbose-ptxas]
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmoe_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "routing.cu", "ffn_simt.cu", "ffn_tc.cu", "ffn_pair.cu", "ffn_nvf4.cu", "ffn_fp8.cu", "router.cu"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")
    return cand


def _compile(src: str, verbose_ptxas: bool, build_dir: str = BUILD, defines=()) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
           *[f"-D{d}" for d in defines], "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    return obj


def build(verbose_ptxas: bool = False, force: bool = False, out: str = LIB, defines=()) -> str:
    """Compile and link the library; returns its path.  Skips work when up to date.

    `out` and `defines` build a variant of the library elsewhere (tile-size
    sweeps pass -D overrides of the kernels' compile-time constants).
    """
    build_dir = BUILD if out == LIB else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    inputs = [os.path.join(CSRC, s) for s in SOURCES] + [
        os.path.join(CSRC, "moe_internal.cuh"), os.path.join(CSRC, "tc_common.cuh"), os.path.join(ROOT, "include", "moe.h"), os.path.abspath(__file__)]
    if not force and not verbose_ptxas and not defines and os.path.exists(out):
        lib_mtime = os.path.getmtime(out)
        if all(os.path.getmtime(p) <= lib_mtime for p in inputs):
            return out
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, build_dir, defines), SOURCES))
    tmp = out + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose_ptxas="--verbose-ptxas" in sys.argv, force="--force" in sys.argv))
