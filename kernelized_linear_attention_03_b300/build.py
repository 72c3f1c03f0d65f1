"""Build ``libkata.so`` (the C-ABI CUDA library) in-tree for sm_103a.

``python -m kernelized_linear_attention_03_b300.build [--force]``.  A stamp file
holding a hash of the sources and flags skips rebuilding an up-to-date library.
"""
import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libkata.so")
STAMP = LIB + ".stamp"
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-shared", "-cudart", "shared",
    "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64"),
    "-I", os.path.join(ROOT, "include"),
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _digest(extra):
    h = hashlib.sha256()
    files = sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")))
    files.append(os.path.join(ROOT, "include", "kata.h"))
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, extra=(), verbose: bool = False) -> str:
    """Compile every CUDA source of the package into libkata.so; return its path."""
    extra = list(extra)
    d = _digest(extra)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == d:
                return LIB
    tmp = LIB + ".tmp"
    cmd = [NVCC] + FLAGS + extra + sources() + ["-o", tmp]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(d)
    return LIB


if __name__ == "__main__":
    args = sys.argv[1:]
    print(build(force="--force" in args, extra=[a for a in args if a != "--force"], verbose=True))
