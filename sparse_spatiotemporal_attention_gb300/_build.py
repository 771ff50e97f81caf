"""Builds the in-tree shared library libskiparse.so for sm_103a with nvcc.

Each .cu file compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically, so the library loads
on a machine without a GPU (calls then return SKIPARSE_ERR_DEVICE).
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
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libskiparse.so")
SYNTH_SRC = os.path.join(CSRC, "synthetic_gen.c")
SYNTH_LIB = os.path.join(LIBDIR, "libsynthetic.so")
SOURCES = ["skiparse_host.cu", "skiparse_fwd.cu", "skiparse_fwd8.cu", "skiparse_bwd.cu", "skiparse_bwd_rows.cu",
           "skiparse_debug.cu", "skiparse_noalloc.cu", "skiparse_proj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libskiparse.so")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build_synthetic(force: bool = False) -> str:
    """Compile the C input generator with the host compiler (no CUDA needed)."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and os.path.exists(SYNTH_LIB) and os.path.getmtime(SYNTH_LIB) >= os.path.getmtime(SYNTH_SRC):
        return SYNTH_LIB
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc:
        raise RuntimeError("no C compiler found for the input generator")
    tmp = SYNTH_LIB + ".tmp"
    _run([cc, "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", tmp, SYNTH_SRC, "-lm"])
    os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile and link; returns the library path. Rebuilds when a source is newer."""
    os.makedirs(LIBDIR, exist_ok=True)
    build_synthetic(force=force)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "skiparse.h"))
    if not force and os.path.exists(LIB):
        lt = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= lt for d in deps):
            return LIB
    nv = nvcc()
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src).replace(".cu", ".o"))
        out = _run([nv] + common + ["-c", src, "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    for obj, out in results:
        if verbose and out.strip():
            print(out, file=sys.stderr)
    tmp = LIB + ".tmp"
    _run([nv] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv))
