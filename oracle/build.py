"""Builds the oracle's shared library (test infrastructure only).

The oracle is compiled with the host C compiler, -O2, no fast-math and no
floating-point contraction, so that every rounding it performs is the one its
source states, on x86-64 and on aarch64 alike.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fused_norm_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_oracle(src: str, out: str) -> str:
    """Compile the C file `src` with the oracle's flags into the shared library `out`."""
    cc = os.environ.get("CC", "gcc")
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    """Compile oracle/fused_norm_oracle.c into oracle/liboracle.so; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_oracle(SRC, LIB)


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
