"""Build libbi.so (the CUDA kernels and their C ABI) in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library next to this file. No CMake, no torch extension
machinery: the library has a plain C ABI and no torch types.

build(debug=True) makes libbi_debug.so instead: the same sources compiled with
BI_DEBUG, whose kernels check every index and coordinate they compute and
record a failure in the device status word (bi_debug_build() returns 1).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbi.so")
OBJDIR_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libbi_debug.so")
SOURCES = ["abi.cu", "gemm_bf16_dense.cu", "gemm_bf16_pair.cu", "gemm_nvfp4.cu", "quantize_nvfp4.cu", "moe.cu", "attention.cu", "rmsnorm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "bi.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    """Compile every .cu for sm_103a and link libbi.so (libbi_debug.so with
    debug=True); returns its path."""
    lib, objdir = (LIB_DEBUG, OBJDIR_DEBUG) if debug else (LIB, OBJDIR)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    extra = list(extra or []) + (["-DBI_DEBUG=1"] if debug else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
