"""Build libdkv.so in-tree for sm_103a (GB300).

Each CUDA translation unit compiles in parallel with nvcc, then one nvcc link
makes the shared library.  IEEE semantics are kept (no --use_fast_math: the
kernels rely on correctly rounded fp32 division, reciprocal and fma).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "lib", "libdkv.so")
# the bounds-checked variant (-DDKV_CHECKED): its own objects and library
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_PATH_CHECKED = os.path.join(HERE, "lib", "libdkv_checked.so")
# host code under AddressSanitizer + UndefinedBehaviorSanitizer (device code
# unchanged), for the argument-validation paths that run without a GPU
BUILD_SAN = os.path.join(HERE, "_build_san")
LIB_PATH_SAN = os.path.join(HERE, "lib", "libdkv_san.so")
HOST_SAN = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
            "-Xcompiler", "-fno-sanitize-recover=all", "-Xcompiler", "-fno-omit-frame-pointer"]
SOURCES = ["api.cu", "classify.cu", "alloc.cu", "pack.cu", "pool.cu", "noalloc.cu", "decode.cu", "attend.cu", "prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(home, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src, os.path.join(CSRC, "dkv_internal.cuh"),
            os.path.join(os.path.dirname(HERE), "include", "dkv.h")]
    return os.path.getmtime(obj) < max(os.path.getmtime(d) for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False, sanitize: bool = False) -> str:
    """Compile the library (the bounds-checked variant when `checked`, the
    host-sanitized one when `sanitize`)."""
    bdir = BUILD_CHECKED if checked else (BUILD_SAN if sanitize else BUILD)
    lib = LIB_PATH_CHECKED if checked else (LIB_PATH_SAN if sanitize else LIB_PATH)
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(bdir, s.replace(".cu", ".o"))
        if force or _stale(obj, src):
            cmd = [nvcc, *ARCH, *FLAGS, *(["-DDKV_CHECKED"] if checked else []), *(HOST_SAN if sanitize else []),
                   "-c", src, "-o", obj]
            if verbose_ptxas:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, results):
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(lib):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([nvcc, *ARCH, "-shared", *(HOST_SAN if sanitize else []), "-o", tmp, *objs, "-lcudart"],
                       check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv,
                sanitize="--sanitize" in sys.argv))
