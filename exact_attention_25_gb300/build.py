"""Builds libfa.so (the C-ABI attention library) in-tree with nvcc for sm_103a only.

Each .cu file under csrc/ is compiled to an object in parallel, then linked into
``exact_attention_25_gb300/libfa.so``.  No cmake, no torch extension machinery: the
library is plain C ABI and is loaded with ctypes.  ``build(checked=True)`` makes the
checked variant ``libfa_checked.so`` (-DFA_CHECKED: every direct global access is tested
against its buffer's extent, see fa_checked_build in include/fa.h) from the same sources.
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
LIB = os.path.join(PKG, "libfa.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libfa_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")
    return path


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(ROOT, "include", "fa.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, verbose_ptxas: bool, checked: bool = False) -> str:
    obj = os.path.join(BUILD_CHECKED if checked else BUILD, os.path.basename(src)[:-3] + ".o")
    if (os.path.exists(obj) and os.path.getmtime(obj) > os.path.getmtime(src)
            and os.path.getmtime(obj) > _headers_mtime()):
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DFA_CHECKED"] if checked else []), "-c", src,
           "-o", obj + ".tmp"]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libfa.so (libfa_checked.so with
    ``checked``); returns its path."""
    bdir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    if force:
        for f in os.listdir(bdir):
            os.remove(os.path.join(bdir, f))
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, checked), srcs))
    if (force or not os.path.exists(lib)
            or max(os.path.getmtime(o) for o in objs) > os.path.getmtime(lib)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Both variants, compiled concurrently."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda c: build(force, checked=c), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                checked="--checked" in sys.argv))
