"""Builds libsplitkv.so in-tree: nvcc for sm_103a, one translation unit per
kernel family, compiled in parallel, linked against the shared CUDA runtime.
``--debug`` builds libsplitkv_debug.so instead (-DSKV_DEBUG=1: the kernels
check their indices, count failures in the plan header and skip the access),
in its own object folder."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsplitkv.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libsplitkv_debug.so")
SOURCES = ["api.cu", "plan.cu", "attn_simt.cu", "attn_tc.cu", "rows.cu", "draft.cu", "noalloc.cu", "proj.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "splitkv.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compiles (if sources changed) and returns the library path."""
    lib, objdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    flags = FLAGS + (["-DSKV_DEBUG=1"] if debug else [])
    if not force and not _stale(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def one(src: str) -> str:
        obj = os.path.join(objdir, src + ".o")
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stdout.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
