"""Compile the CPU oracle (gemm_oracle.c) into oracle/liboracle.so.

TEST INFRASTRUCTURE ONLY: the library built here is loaded by the tests, the
smoke check and the benchmark's CPU-baseline leg, never by the product path.

Plain gcc, portable flags only (the same source builds on x86_64 and on
aarch64): no -march=native, no vector intrinsics.  -ffp-contract=off keeps a
multiply and an add as two roundings on every machine.  OpenMP is used when the
compiler has it; without it the oracle runs on one thread.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def _stale() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False, verbose: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source; return its path."""
    if not force and not _stale():
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    attempts = [BASE_FLAGS + ["-fopenmp"], BASE_FLAGS]
    last = None
    for flags in attempts:
        cmd = [cc] + flags + [SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
        last = r.stderr
    raise RuntimeError("oracle build failed:\n" + (last or ""))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
