"""In-tree build of libmla_sparse.so (nvcc, sm_103a only)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, "mla_sparse_fwd.cu"), os.path.join(CSRC, "lightning_indexer.cu"),
           os.path.join(CSRC, "cache_write.cu"), os.path.join(CSRC, "mla_prolog.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(ROOT, "include", "mla_sparse.h"),
                  os.path.join(ROOT, "include", "mla_indexer.h"), os.path.join(ROOT, "include", "mla_cache.h"),
                  os.path.join(ROOT, "include", "mla_prolog.h")]
LIB_PATH = os.path.join(HERE, "libmla_sparse.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "--threads", "4"]


def nvcc() -> str:
    cand = os.path.join(cuda_home(), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def cuda_home() -> str:
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def link_flags() -> list:
    """The CUDA runtime and driver API (tensor-map encoding), found through the toolkit's library directory."""
    lib = os.path.join(cuda_home(), "lib64")
    return ["-L" + lib, "-Xlinker", "-rpath=" + lib]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library unless it is newer than all of its sources."""
    if not force and os.path.exists(LIB_PATH):
        t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(d) <= t for d in DEPS):
            return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-o", tmp] + SOURCES + link_flags()
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
