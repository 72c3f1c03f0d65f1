"""Build ``libkata.so`` (the C-ABI CUDA library) in-tree for sm_103a.

``python -m kernelized_linear_attention_03_b300.build [--force]``.  A stamp file
holding a hash of the sources and flags skips rebuilding an up-to-date library.
"""
import glob
import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

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
    "-I", os.path.join(ROOT, "include"),
]
LINK = ["-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "shared",
        "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")]
OBJ = os.path.join(PKG, "_build")


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
    h.update(" ".join(FLAGS + LINK + extra).encode())
    return h.hexdigest()


def build(force: bool = False, extra=(), verbose: bool = False) -> str:
    """Compile every CUDA source of the package into libkata.so; return its path."""
    extra = list(extra)
    d = _digest(extra)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == d:
                return LIB
    os.makedirs(OBJ, exist_ok=True)
    objs = [os.path.join(OBJ, os.path.basename(src)[:-3] + ".o") for src in sources()]

    def compile_one(src, obj):
        cmd = [NVCC] + FLAGS + extra + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        subprocess.run(cmd, check=True)

    # one nvcc per translation unit, in parallel; then one link
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as pool:
        for f in [pool.submit(compile_one, s_, o_) for s_, o_ in zip(sources(), objs)]:
            f.result()
    tmp = LIB + ".tmp"
    subprocess.run([NVCC] + LINK + objs + ["-o", tmp], check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(d)
    return LIB


if __name__ == "__main__":
    args = sys.argv[1:]
    print(build(force="--force" in args, extra=[a for a in args if a != "--force"], verbose=True))
