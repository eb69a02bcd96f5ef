"""Build the CPU oracle (plain C11) into oracle/_build/liboracle.so with gcc.

Test infrastructure: the oracle is the independent checker of the CUDA
library and is never linked into it.  No fast-math and no FMA contraction,
so each float operation in the oracle is one IEEE operation on x86-64 and on
Arm alike.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8w_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
          "-ffp-contract=off", "-fno-strict-aliasing", "-pthread",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
