"""Compile the fp64 CPU oracle into ``oracle/libkata_oracle.so``.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use the oracle.  Plain ``g++ -O2`` without fast-math, so the fp64
arithmetic follows the source order.
"""
import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kata_oracle.cpp")
LIB = os.path.join(HERE, "libkata_oracle.so")
STAMP = LIB + ".stamp"
CMD = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
       "-pthread", SRC, "-o", LIB]


def _digest() -> str:
    h = hashlib.sha256()
    with open(SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(CMD).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Build the oracle library if missing or stale; return its path."""
    d = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == d:
                return LIB
    subprocess.run(CMD, check=True)
    with open(STAMP, "w") as f:
        f.write(d)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
