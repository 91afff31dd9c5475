"""Build libkda_gb300.so (CUDA kernels + C ABI) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process in parallel, then
linked into ``kda_linear_attention_gb300/libkda_gb300.so``.  Usage:

    python -m kda_linear_attention_gb300.build [--force] [--verbose] [--debug]
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda_gb300.so")
# debug build: the kernels' index checks compiled in (KDA_DEBUG); selected at
# run time with KDA_GB300_DEBUG=1
OBJ_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libkda_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda_gb300")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(force: bool, lib: str = LIB) -> bool:
    if force or not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps.append(os.path.join(ROOT, "include", "kda.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link the library; returns its
    path.  debug=True builds libkda_gb300_debug.so with the kernels' index
    checks (-DKDA_DEBUG) instead."""
    lib_path, obj_dir = (LIB_DEBUG, OBJ_DEBUG) if debug else (LIB, OBJ)
    if not _stale(force, lib_path):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    nv = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DKDA_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nv] + ARCH + flags + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [nv] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug", action="store_true",
                    help="build libkda_gb300_debug.so with the kernels' index checks")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug=a.debug))
