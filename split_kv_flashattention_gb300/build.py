"""Build libfa_splitkv.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into split_kv_flashattention_gb300/lib/
libfa_splitkv.so with the CUDA runtime linked statically and only the fa_*
C symbols exported.  Usage: python -m split_kv_flashattention_gb300.build

--debug builds lib/libfa_splitkv_debug.so from the same sources with
-DFA_DEBUG (objects under _build_debug/): every global index the kernels
use is checked first, and a failed check records FA_ERR_DEVICE_BOUNDS in the
device error word and skips the access.  The binding loads it when the
environment variable FA_SPLITKV_DEBUG is 1.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libfa_splitkv.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(LIBDIR, "libfa_splitkv_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC] + list(extra)


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
        os.path.join(ROOT, "include", "fa_splitkv.h")]


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.basename(src)[:-3] + ".o")
    newest_dep = max(os.path.getmtime(h) for h in _headers() + [src])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest_dep and not verbose_ptxas:
        return obj
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DFA_DEBUG"] if debug else [])
    cmd = [nvcc()] + _flags(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _machine_stamp(build_dir: str = BUILD, lib: str = LIB):
    """Objects (and the library) built on another host architecture are
    discarded."""
    stamp = os.path.join(build_dir, "host_arch.txt")
    arch = platform.machine()
    old = open(stamp).read().strip() if os.path.exists(stamp) else None
    if old != arch:
        for f in os.listdir(build_dir):
            if f.endswith((".o", ".tmp", ".map")):
                os.remove(os.path.join(build_dir, f))
        for f in (lib, lib + ".tmp"):
            if os.path.exists(f):
                os.remove(f)
        with open(stamp, "w") as f:
            f.write(arch + "\n")


def build(verbose_ptxas: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    build_dir = BUILD_DEBUG if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    _machine_stamp(build_dir, lib)
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), srcs))
    vers = os.path.join(build_dir, "exports.map")
    with open(vers, "w") as f:
        f.write("{ global: fa_*; local: *; };\n")
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return lib
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + [
        "-Xlinker", f"--version-script={vers}", "-Xlinker", "--exclude-libs,ALL"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
