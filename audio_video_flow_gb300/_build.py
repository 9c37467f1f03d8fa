"""Builds libh3.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit is compiled in parallel into _build/, then linked with
nvcc into audio_video_flow_gb300/libh3.so (CUDA runtime linked statically).
build(bounds=True) builds the bounds-checked variant instead
(-DH3_BOUNDS_CHECK=1, objects in _build_bounds/, libh3_bounds.so): every
checked global access of the kernels first tests that it lies inside the
buffer the call's arguments describe, and reports H3_ERR_BOUNDS instead.
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
LIB = os.path.join(PKG, "libh3.so")
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libh3_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
          "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(nvcc: str, src: str, extra, out_dir: str = BUILD) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(out_dir, os.path.basename(src) + ".log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    return obj


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "h3.h"))
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, extra_flags=(), verbose: bool = False, bounds: bool = False) -> str:
    lib, out_dir = (LIB_BOUNDS, BUILD_BOUNDS) if bounds else (LIB, BUILD)
    if not force and not extra_flags and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    flags = list(extra_flags) + (["-DH3_BOUNDS_CHECK=1"] if bounds else [])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, flags, out_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr[-4000:])
    os.replace(tmp, lib)
    if verbose:
        for s in srcs:
            print(open(os.path.join(out_dir, os.path.basename(s) + ".log")).read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds="--bounds" in sys.argv))
