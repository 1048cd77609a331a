"""Builds libmk.so (the decode megakernel and its C ABI) for sm_103a with nvcc.

Each translation unit compiles in parallel; the shared library is written in
the package directory, where the Python binding loads it."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SOURCES = ["mk_api.cpp", "mk_sched.cpp", "mk_shape_tiny.cu", "mk_shape_small.cu", "mk_shape_full.cu",
           "mk_shape_dense.cu", "mk_static_ws.cu", "mk_service.cpp", "mk_gpu_step.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def source_hash() -> str:
    """sha256 over the kernel sources and the public header (identifies the
    kernel a recorded profile was taken on)."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)) + ["../../include/mk.h"]:
        path = os.path.join(CSRC, name)
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def _nvcc() -> str:
    return os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    common = [_nvcc(), "-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2",
              "-I", os.path.join(HERE, "..", "include")]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_verbose or verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    out = os.path.join(HERE, "libmk.so")
    cmd = [_nvcc(), "-shared", *ARCH, "-o", out + ".tmp", *objs, "-lcudart"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
