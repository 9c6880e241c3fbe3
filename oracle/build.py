"""Build step for the oracle's shared library (test infrastructure only).

Compiles ``oracle.c`` with the host C compiler into ``liboracle.so`` beside
it.  The flags keep IEEE binary32 arithmetic exact as the C standard states
it: no fast-math, no contraction of a*b+c into fused operations (there are
none in the sums, but the flag keeps it so), no finite-math assumptions.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-pthread"]


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
