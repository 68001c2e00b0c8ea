"""Build step of the CUDA library: one nvcc invocation for sm_103a.

Produces ``dense_bf16_gemm_02_gb300/_build/libhk_gemm.so`` (in-tree), which
exports the C-ABI declared in ``include/hk_gemm.h``. The CUDA runtime is linked
statically, so loading the library needs no GPU and no LD_LIBRARY_PATH.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libhk_gemm.so")
SOURCES = [os.path.join(CSRC, "hk_gemm.cu"), os.path.join(CSRC, "hk_attention.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "hk_gemm.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def compile_command(src: str, obj: str, verbose_ptxas: bool = False) -> list[str]:
    cmd = [nvcc_path(), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17", "-c",
           "-Xcompiler", "-fPIC,-O2", "-o", obj, src]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def link_command(objs: list[str], out: str) -> list[str]:
    return [nvcc_path(), *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", out, *objs]


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library unless it is newer than every source. The
    translation units compile in parallel, then one link."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(f) for f in DEPENDS)):
        return LIB_PATH
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD_DIR, os.path.splitext(os.path.basename(s))[0] + tag + ".o") for s in SOURCES]
    procs = [subprocess.Popen(compile_command(s, o, verbose_ptxas)) for s, o in zip(SOURCES, objs)]
    codes = [pr.wait() for pr in procs]
    try:
        if any(codes):
            raise subprocess.CalledProcessError(next(c for c in codes if c), "nvcc -c")
        tmp = LIB_PATH + tag
        subprocess.run(link_command(objs, tmp), check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas=True))
