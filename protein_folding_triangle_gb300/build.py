"""In-tree build of libtriattn (nvcc, sm_103a only).

Each translation unit is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3`` and linked
into ``_build/libtriattn_<machine>.so`` next to this file.  No cmake, no
torch extension machinery: the library exports a plain C ABI
(include/triattn.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "noalloc.cu", "module.cu", "trimul.cu", "gemm.cu"]
HEADERS = ["ptx.cuh", "kernels.cuh", "pairops.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtriattn")
    return exe


def lib_path() -> str:
    return os.path.join(BUILD, f"libtriattn_{platform.machine()}.so")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libtriattn if any source is newer than the library."""
    out = lib_path()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "triattn.h"), __file__]
    if not force and not _stale(out, deps):
        return out
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    objs = [os.path.join(BUILD, f"{os.path.splitext(s)[0]}_{platform.machine()}.o") for s in SOURCES]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [exe] + NVCC_FLAGS + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    tmp = out + f".tmp{os.getpid()}"
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(exe))), "lib64")
    cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs + ["-L", cuda_lib, "-Xlinker", "-rpath=" + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
