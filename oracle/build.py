"""Compile the C oracle (oracle.c) into oracle/liboracle.so with gcc.

Test infrastructure: the oracle is built so that the tests, the smoke check
and the benchmark's CPU-baseline leg can load it; the CUDA library never does.
Plain, portable flags only (the same source builds on x86_64 and aarch64);
-ffp-contract=off keeps a*b+c as two roundings on every machine.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Build the shared library if it is missing or older than its source."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
