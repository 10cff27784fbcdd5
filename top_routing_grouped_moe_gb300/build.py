"""Builds the CUDA library in-tree: every csrc/*.cu is compiled for sm_103a
in parallel and linked (static CUDA runtime) into lib/libmoe_gb300.so.

    python -m top_routing_grouped_moe_gb300.build [--force]
"""
from __future__ import annotations

import glob
import hashlib
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libmoe_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


STAMP = LIB + ".stamp"


def _fingerprint() -> str:
    """Hash of every source file's path and contents plus the flags."""
    h = hashlib.sha256()
    for p in sorted(_deps()):
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


_GEMM_COMMON = ["gemm.cuh", "gemm_host.cuh", "ptx.cuh", "common.cuh", "internal.h"]


def _kernel_sources(kernel: str):
    """csrc files the named kernel (a launch name of moe_timing_name) is
    compiled and launched from."""
    if kernel.startswith("gemm_router"):
        files = _GEMM_COMMON + ["gemm_router.cu"]
    elif kernel.startswith("gemm_mx"):
        files = _GEMM_COMMON + ["gemm_mx.cu"]
    elif kernel.startswith(("gemm_gate_up", "gemm_down")):
        files = _GEMM_COMMON + ["gemm_fwd.cu"]
    elif kernel.startswith(("gemm_dgrad", "gemm_wgrad")):
        files = _GEMM_COMMON + ["gemm_bwd.cu", "group_maps.cu"]
    elif kernel == "group_maps":
        files = ["group_maps.cu", "gemm_host.cuh", "gemm.cuh", "ptx.cuh", "common.cuh", "internal.h"]
    elif kernel.startswith("mx_") or kernel.endswith("_mx"):
        files = ["mxfp8.cu", "route.cu", "common.cuh", "internal.h"]
    else:
        files = ["route.cu", "common.cuh", "internal.h"]
    return [os.path.join(CSRC, f) for f in files]


def _strip_comments(src: str) -> str:
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return " ".join(src.split())


def kernel_fingerprint(kernel: str) -> str:
    """Hash of the code (comments and layout removed) of the sources one kernel
    is built and launched from, plus the compiler flags: a profile of that
    kernel stays valid across edits elsewhere in the library."""
    h = hashlib.sha256()
    for p in _kernel_sources(kernel):
        h.update(os.path.basename(p).encode())
        with open(p) as f:
            h.update(_strip_comments(f.read()).encode())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()[:32]


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _fingerprint()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_fingerprint())
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    print(build(force=force, verbose="-v" in sys.argv))
