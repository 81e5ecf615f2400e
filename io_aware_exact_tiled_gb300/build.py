"""Builds libfa.so in-tree from csrc/ with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into a shared
library with the CUDA runtime linked statically (no driver library at link
time: tensor maps are encoded through the runtime's driver entry point).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd_t1.cu", "fa_bwd.cu", "fa_noalloc.cu", "fa_decode.cu", "fa_fwd_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _compile(src: str, extra, build_dir: str = BUILD_DIR) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, extra_flags=(), lib: str = LIB, build_dir: str = BUILD_DIR) -> str:
    """Compile csrc/*.cu and link the library (libfa.so unless `lib` says
    otherwise, e.g. a debug variant built with extra flags); returns its path."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fa.h")]
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= t for d in deps):
            return lib
    os.makedirs(build_dir, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags), build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


DEBUG_LIB = os.path.join(PKG, "libfa_debug.so")


def build_debug(force: bool = False) -> str:
    """Debug variant for the give-up test: short (0.2 s) device wait limit and
    one withheld "P ready" arrival per kernel (FA_DEBUG_DROP_ARRIVE)."""
    return build(force, ("-DFA_DEBUG_DROP_ARRIVE", "-DFA_WAIT_LIMIT_NS=200000000ull"), DEBUG_LIB,
                 os.path.join(PKG, "_build_debug"))


if __name__ == "__main__":
    print(build(force=True))
