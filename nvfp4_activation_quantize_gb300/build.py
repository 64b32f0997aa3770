"""Build libh3q.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit under ``csrc/`` is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a``, then linked into
``_build/libh3q.so`` (CUDA runtime linked statically, so the library loads
without a GPU).  ``-fmad=false`` and the absence of fast-math keep every
binary32 operation a separately rounded IEEE operation, which the kernels'
bit-exactness relies on.  ptxas resource usage is kept in
``_build/ptxas.log``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libh3q.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "h3q.h")

SOURCES = ["h3q_api.cu", "quantize.cu", "adaln.cu", "swiglu.cu", "dequantize.cu", "amax.cu",
           "residual.cu", "qkv.cu", "host_pipeline.cu", "gemm_swiglu.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libh3q.so")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [HEADER, __file__]
    return [p for p in deps if os.path.isfile(p)]


def is_fresh() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libh3q.so unless it is already newer than its sources."""
    if not force and is_fresh():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(len(SOURCES)) as pool:
        results = list(pool.map(compile_one, SOURCES))
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as log:
        for (_, err), src in zip(results, SOURCES):
            log.write(f"== {src}\n{err}\n")
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
