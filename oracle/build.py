"""Compile the CPU oracle (test infrastructure) with gcc into oracle/_build/.

The oracle is a checker, not part of the product path: the tests, the
package's smoke check and the benchmark's CPU baseline are its only users.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libspecoracle.so")

# IEEE double everywhere: no fast-math, no contraction of a*b+c into an FMA
# (gcc contracts by default on aarch64), so x86 and Arm hosts agree bit for bit.
CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm", "-lpthread"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
