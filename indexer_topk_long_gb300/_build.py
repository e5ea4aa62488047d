"""In-tree build of libltk.so with nvcc for sm_103a (no CMake).

Each ``csrc/*.cu`` compiles to an object under ``_build/`` in parallel; the
objects link into ``indexer_topk_long_gb300/libltk.so`` (static cudart, no
libcuda link: the one driver entry point used, the tensor-map encoder, is
fetched at run time).  An object is rebuilt when its source or a header is
newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libltk.so")
HEADERS = [*(os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cuh")),
           os.path.join(ROOT, "include", "ltk.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "--expt-relaxed-constexpr"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def _stale(src: str, obj: str) -> bool:
    t = _mtime(obj)
    return t < 0 or any(_mtime(x) > t for x in [src, *HEADERS])


def _compile(src: str, extra: list[str], verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if not _stale(src, obj):
        return obj
    tmp = obj + ".tmp.o"
    cmd = [nvcc(), *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", tmp]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    os.replace(tmp, obj)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link libltk.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    if force:
        for s in srcs:
            o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
            if os.path.exists(o):
                os.remove(o)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose or ptxas_verbose), srcs))
    if force or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


def ensure_built() -> str:
    srcs = sources()
    if not os.path.exists(LIB) or any(_mtime(s) > _mtime(LIB) for s in srcs + HEADERS):
        return build()
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
