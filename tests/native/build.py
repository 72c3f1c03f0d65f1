"""Build the tcgen05 self-test library (test infrastructure) in-tree for sm_103a."""
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
SRC = os.path.join(HERE, "tc_selftest.cu")
LIB = os.path.join(HERE, "libkata_tc_selftest.so")
DEPS = [SRC, os.path.join(ROOT, "kernelized_linear_attention_03_b300", "csrc", "tc_primitives.cuh")]
CMD = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
       "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
       "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", SRC, "-o", LIB]


def build(force=False):
    h = hashlib.sha256(" ".join(CMD).encode())
    for f in DEPS:
        h.update(open(f, "rb").read())
    stamp = LIB + ".stamp"
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == h.hexdigest():
        return LIB
    subprocess.run(CMD, check=True)
    with open(stamp, "w") as f:
        f.write(h.hexdigest())
    return LIB


if __name__ == "__main__":
    print(build(force=True))
