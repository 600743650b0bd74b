"""Build ``libdecgemm.so`` in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically. The same sources
compiled with -DDEC_DEBUG link into ``libdecgemm_debug.so``, whose kernels
check every computed index against the extent of the buffer it addresses
(a failed check is reported by dec_sync_check as DEC_EBOUNDS; the access is
skipped). Run as ``python -m moe_decode_gemm_gb300.build`` or call
``build()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdecgemm.so")
DEBUG_LIB = os.path.join(HERE, "libdecgemm_debug.so")
ROOT = os.path.dirname(HERE)

SOURCES = ["api.cu", "k_linear.cu", "k_moe.cu", "k_tc.cu", "k_gemv.cu", "k_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(ROOT, "include", "decgemm.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, extra, objdir=OBJ) -> str:
    obj = os.path.join(objdir, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(path)
            and os.path.getmtime(obj) >= _headers_mtime()):
        return obj
    cmd = [nvcc()] + ARCH + FLAGS + list(extra) + ["-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def _link(lib: str, objs, force: bool):
    if (not os.path.exists(lib) or force
            or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs)):
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)


def build(verbose_ptxas: bool = False, force: bool = False, debug: bool = True) -> str:
    """Build the library (and, with debug, its index-checking twin); returns
    the library's path."""
    dbg_dir = os.path.join(OBJ, "debug")
    os.makedirs(dbg_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if force:
        for d in (OBJ, dbg_dir):
            for f in os.listdir(d):
                if f.endswith(".o"):
                    os.remove(os.path.join(d, f))
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    jobs = [(s, extra, OBJ) for s in srcs]
    if debug:
        jobs += [(s, extra + ["-DDEC_DEBUG"], dbg_dir) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(*j), jobs))
    _link(LIB, objs[:len(srcs)], force)
    if debug:
        _link(DEBUG_LIB, objs[len(srcs):], force)
    return LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, force="-f" in sys.argv))
