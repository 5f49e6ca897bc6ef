"""Compile libpv.so (the CUDA library) in-tree with nvcc for sm_103a."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
# Every translation unit of libpv.so: the block-tile voxelizer, the unordered
# voxelizer, centroid downsampling, the host side with the C ABI, and farthest
# point sampling (kernel and entry); pv_device.cuh is the kernels' shared code.
SRCS = [os.path.join(CSRC, f) for f in ("pv_ordered.cu", "pv_ordered_half.cu", "pv_unordered.cu", "pv_downsample.cu",
                                         "pv_downsample_half.cu", "pv_host.cu", "pv_fps.cu")]
HEADERS = [os.path.join(CSRC, "pv_device.cuh")]
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libpv.so")

# IEEE binary32 semantics are part of the contract: no fast-math, no flush of
# subnormals, correctly rounded division, no multiply-add contraction.
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
    "-Xcompiler", "-fPIC", "-shared",
]
COMPILE_FLAGS = [f for f in NVCC_FLAGS if f != "-shared"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def sources():
    return [*SRCS, *HEADERS, os.path.join(INCLUDE, "pv.h")]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build(out: str = LIB, extra=(), verbose: bool = False) -> str:
    """Compile every translation unit (in parallel) and link the library; returns its path."""
    from concurrent.futures import ThreadPoolExecutor

    objs = [f"{out}.{os.path.splitext(os.path.basename(src))[0]}.o" for src in SRCS]

    def compile_one(src, obj):
        cmd = [nvcc_path(), *COMPILE_FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
        return subprocess.run(cmd, capture_output=True, text=True)

    with ThreadPoolExecutor(max_workers=len(SRCS)) as ex:
        results = list(ex.map(compile_one, SRCS, objs))
    for res in results:
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
        if verbose:
            print(res.stdout + res.stderr)
    tmp = out + ".tmp"
    link = subprocess.run([nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp],
                          capture_output=True, text=True)
    for o in objs:
        if os.path.exists(o):
            os.remove(o)
    if link.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + link.stdout + link.stderr)
    os.replace(tmp, out)
    return out
