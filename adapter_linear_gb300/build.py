"""Build the CUDA library in-tree: nvcc for sm_103a, one object per .cu file
compiled in parallel, linked into adapter_linear_gb300/liblora_linear.so; and the
checked build (LORA_CHECK defined: every gathered index range-checked in the
kernels) into adapter_linear_gb300/liblora_linear_check.so.

Usage: python -m adapter_linear_gb300.build [--check-only]   (or __graft_entry__.build()).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblora_linear.so")
OBJ_CHECK = os.path.join(HERE, "_build_check")
LIB_CHECK = os.path.join(HERE, "liblora_linear_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include"), *ARCH]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps.append(os.path.join(ROOT, "include", "lora_linear.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=(), check: bool = False) -> str:
    """Compile and link one library; check=True: the LORA_CHECK build."""
    obj_dir, lib = (OBJ_CHECK, LIB_CHECK) if check else (OBJ, LIB)
    if check:
        extra_flags = (*extra_flags, "-DLORA_CHECK")
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(verbose: bool = False) -> None:
    """Both libraries, at the same time (twice the translation units in flight)."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, verbose), ex.submit(build, verbose, (), True)]:
            f.result()


if __name__ == "__main__":
    v = "-v" in sys.argv
    flags = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    if "--check-only" in sys.argv:
        print(build(verbose=v, check=True))
    elif flags:
        print(build(verbose=True, extra_flags=flags))
    else:
        build_all(verbose=v)
        print(LIB, LIB_CHECK)
