"""Compile the C oracle into oracle/liboracle.so (plain gcc, fp64, OpenMP).

No fast-math: the oracle keeps IEEE double semantics so that its sums are
the plain definitions.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "isd_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    return (not os.path.exists(LIBRARY)
            or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIBRARY + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
               "-fvisibility=hidden", "-Wall", "-Wextra", SOURCE, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
