"""Compile the fp64 CPU oracle (``gdn_oracle.c``) into ``libgdn_oracle.so``.

Test infrastructure: the library built here is loaded only by the test suite,
the smoke check and the benchmark's CPU-baseline leg.  Plain gcc, OpenMP when
the compiler accepts it, no architecture-specific flags (the same source
builds on x86_64 and aarch64).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
LIB = os.path.join(HERE, "libgdn_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
