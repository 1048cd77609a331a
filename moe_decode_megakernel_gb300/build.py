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
SOURCES = ["mk_api.cpp", "mk_sched.cpp", "mk_static_ws.cu", "mk_service.cpp", "mk_gpu_step.cu"]
# the compiled model shapes (hidden, n_q, n_kv, head_dim, n_experts, top_k, inter,
# page_size; the same table as kShapes in mk_api.cpp) and kernel modes (KernelMode):
# mk_shape.cu is compiled once per pair
SHAPES = {"tiny": "256,4,2,64,16,4,128,16", "small": "1024,16,2,64,32,4,512,64",
          "dense": "1024,16,2,64,1,1,2048,64", "full": "2048,32,4,128,128,8,768,64"}
MODES = 8
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

    def compile_one(unit) -> str:
        src, defs, name = unit
        obj = os.path.join(BUILD, name + ".o")
        cmd = common + defs + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_verbose or verbose:
            print(r.stderr)
        return obj

    units = [(src, [], os.path.splitext(src)[0]) for src in SOURCES]
    for shape, dims in SHAPES.items():
        for mode in range(MODES):
            fn = f"launch_{shape}_{mode}"
            defs = [f"-DMK_DIM{i}={v}" for i, v in enumerate(dims.split(","))]  # nvcc splits -D at commas
            units.append(("mk_shape.cu", defs + [f"-DMK_MODE={mode}", f"-DMK_LAUNCH_FN={fn}"],
                          f"mk_shape_{shape}_{mode}"))
    with cf.ThreadPoolExecutor(max_workers=min(len(units), max(4, os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, units))
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
