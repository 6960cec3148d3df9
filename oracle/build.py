"""Compile the C oracle into ``oracle/_build/librn_oracle.so`` with gcc.

Test infrastructure: the oracle is built so that tests, the smoke check and
the benchmark's CPU-baseline leg can call it; the product never loads it.
Flags keep fp64 arithmetic exactly as written (no contraction into FMA, no
fast-math reassociation), so x86 and Arm hosts give the same bits.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rmsnorm_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "librn_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math"]


def compile_c(src_path: str, out_path: str) -> str:
    """Compile one C file into a shared library at out_path (atomic rename)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, src_path, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_c(SRC, LIB)


if __name__ == "__main__":
    print(build(force=True))
