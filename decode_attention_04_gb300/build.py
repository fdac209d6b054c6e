"""Builds libfd.so in-tree with nvcc for sm_103a (GB300).

The CUDA and C++ translation units compile in parallel; the link uses the
static CUDA runtime, so the library needs nothing from torch. Run as a module
or call ``build()``; the result is ``decode_attention_04_gb300/libfd.so``,
plus, where Python headers exist, the small CPython module ``_fdfast`` that
calls its per-call entry points with less host overhead than ctypes.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libfd.so"
BUILD_DIR = PKG / "_build"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", str(INCLUDE), "-I", str(CSRC)] + ARCH
SOURCES = ["fd_kernels.cu", "fd_umma.cu", "fd_api.cpp", "fd_noalloc.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfd.so")


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = ([CSRC / s for s in SOURCES] + list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.c")) +
            list(INCLUDE.glob("*.h")) + [Path(__file__)])
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not _stale():
        return LIB
    BUILD_DIR.mkdir(exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = BUILD_DIR / (src + ".o")
        objs.append(obj)
        cmd = [cc, *COMMON, "-c", str(CSRC / src), "-o", str(obj)]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        log = open(BUILD_DIR / (src + ".log"), "w")
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, p, log in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    if failed:
        msgs = "\n".join((BUILD_DIR / (s + ".log")).read_text()[-4000:] for s in failed)
        raise RuntimeError(f"nvcc failed for {failed}:\n{msgs}")
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    subprocess.run([cc, "-shared", *ARCH, "-o", str(tmp), *map(str, objs), "-cudart", "static"], check=True)
    os.replace(tmp, LIB)
    build_fast(verbose=verbose)
    if verbose:
        print((BUILD_DIR / "fd_kernels.cu.log").read_text())
    return LIB


def fast_path() -> Path:
    import sysconfig
    return PKG / ("_fdfast" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_fast(verbose: bool = False) -> Path | None:
    """The CPython entries of fd_pyfast.c, linked to libfd.so beside them
    (optional: without Python headers the package calls libfd.so through
    ctypes alone)."""
    import sysconfig
    inc = sysconfig.get_paths().get("include")
    if not inc or not (Path(inc) / "Python.h").exists():
        if verbose:
            print("Python headers not found: the ctypes route serves every call")
        return None
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc:
        return None
    out = fast_path()
    tmp = out.with_suffix(f".tmp{os.getpid()}")
    cmd = [cc, "-shared", "-fPIC", "-O2", "-I", inc, "-I", str(INCLUDE), str(CSRC / "fd_pyfast.c"), "-L", str(PKG),
           "-lfd", "-Wl,-rpath,$ORIGIN", "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if verbose:
            print("fd_pyfast.c did not build (the ctypes route serves every call):\n" + r.stderr[-2000:])
        return None
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
