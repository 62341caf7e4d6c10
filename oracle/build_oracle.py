"""Compile the CPU oracle (oracle/aq_oracle.c) into oracle/libaq_oracle.so.

Test infrastructure: the oracle is built so that tests, the smoke check and
the benchmark's CPU-baseline leg can load it.  Plain gcc, no CUDA.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "aq_oracle.c")
HDR = os.path.join(HERE, "aq_oracle.h")
LIB = os.path.join(HERE, "libaq_oracle.so")

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
          "-Wall", "-Wextra", "-fPIC", "-shared"]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    built = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > built for p in (SRC, HDR))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
