"""Builds libmoeroute.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel into ``_build/`` and linked into
``combine_moe_route_05_gb300/libmoeroute.so``.  Rebuilds only when a source or
header is newer than the library.
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoeroute.so")
SOURCES = ["route.cu", "layout.cu", "rows.cu", "api.cu", "layout_static.cu", "w2_gemm.cu"]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src, extra):
    obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC] + ARCH + FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(force=False, verbose=False, extra=()):
    if not force and not extra and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, log in results:
        if verbose or rc != 0:
            sys.stderr.write("== %s (rc=%d)\n%s" % (src, rc, log))
    if failed:
        raise RuntimeError("nvcc failed for: %s" % ", ".join(r[0] for r in failed))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [r[1] for r in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force=True, verbose=v, extra=["-Xptxas", "-v"] if v else []))
