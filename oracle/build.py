"""Build the CPU oracle (plain C, host only) into oracle/libtmap_oracle.so.

Test infrastructure: the oracle is compiled so that the test suite and the benchmark's CPU
baseline can call it; the product library never links it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tmap_oracle.c")
LIB = os.path.join(HERE, "libtmap_oracle.so")

# No -ffast-math and no contraction: the fp32 reduce-add must be one IEEE binary32 add.
CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math"]


def build(force: bool = False) -> str:
    deps = [SRC, os.path.join(HERE, "tmap_oracle.h")]
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in deps):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
