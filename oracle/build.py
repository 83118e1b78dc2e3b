"""Compile the CPU oracle (plain C, double precision) into oracle/_build/liboracle.so.

Test infrastructure: the test suite, the smoke check and the benchmark's CPU
baseline leg load the result; the product library never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
          "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """Compile one C source file into the shared library ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than oracle.c; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force=True))
