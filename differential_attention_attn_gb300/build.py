"""Build libdiffattn.so in-tree with nvcc for sm_103a (no cmake, no torch).

Each .cu file is compiled to an object in parallel, then linked as a shared
library against the static CUDA runtime (the driver's cuTensorMapEncodeTiled
is looked up at run time, so the library loads on hosts without a driver).
Outputs land next to this file, under _build/ and libdiffattn.so, both
git-ignored.  build(debug=True) makes the bounds-checked variant instead
(-DDIFFATTN_DEBUG: every kernel checks its tensor-memory, shared-memory and
global accesses and reports a failed check through the status word) as
libdiffattn_debug.so under _build_debug/.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdiffattn.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libdiffattn_debug.so")
SOURCES = ["api.cu", "fwd_bf16_sm103.cu", "fwd_f32.cu", "headnorm.cu", "splitkv.cu",
           "noalloc.cu", "bwd_bf16_sm103.cu", "fwd_d128_sm103.cu", "bwd_d128_sm103.cu",
           "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool, debug: bool = False) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    if debug:
        f += ["-DDIFFATTN_DEBUG"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> tuple[str, str]:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *_flags(verbose_ptxas, debug), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "diffattn.h"))
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(BUILD_DEBUG if debug else BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), SOURCES))
    if verbose_ptxas:
        for _, log in results:
            sys.stdout.write(log)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
