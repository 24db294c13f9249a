"""Builds libadaln.so in-tree for GB300 (sm_103a): one nvcc per translation unit, in
parallel, then one link. No CMake, no torch extension machinery. build(debug=True) makes
libadaln_debug.so, the same sources compiled with -DADALN_DEBUG (every kernel checks each
computed index before the access; see adaln_debug_read in include/adaln.h)."""
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
BUILD = os.path.join(ROOT, "_build", "adaln")
LIB = os.path.join(PKG, "libadaln.so")
DEBUG_BUILD = os.path.join(ROOT, "_build", "adaln_debug")
DEBUG_LIB = os.path.join(PKG, "libadaln_debug.so")
SOURCES = ["adaln.cu", "fwd.cu", "bwd.cu", "schedule.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags(verbose_ptxas: bool = False) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "-I", CSRC]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _inputs() -> list:
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "adaln.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    lib_path, objdir = (DEBUG_LIB, DEBUG_BUILD) if debug else (LIB, BUILD)
    if not force and not verbose_ptxas and up_to_date(lib_path):
        return lib_path
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    extra = ["-DADALN_DEBUG"] if debug else []

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc] + flags(verbose_ptxas) + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + ".tmp%d" % os.getpid()
    subprocess.check_call([cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results])
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
