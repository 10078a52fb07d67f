"""Compile the CPU oracle (test infrastructure) into oracle/libflint_oracle.so.

Plain gcc, no fast-math and no contraction of a*b+c: the oracle keeps IEEE
FP32 and double semantics, one rounding per written operation.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "flint_oracle.c")
LIB = os.path.join(HERE, "libflint_oracle.so")
# The same source with -fopenmp: output rows split over the host's threads
# (each row still summed in index order by one thread, so the same bits).
LIB_OMP = os.path.join(HERE, "libflint_oracle_omp.so")


def _compile(out: str, extra) -> None:
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-Wall", "-Wextra", "-Wno-unknown-pragmas", *extra, "-o", out + ".tmp", SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        _compile(LIB, [])
    return LIB


def build_omp(force: bool = False):
    """Path of the OpenMP build, or None where the compiler has no OpenMP."""
    if force or not os.path.exists(LIB_OMP) or os.path.getmtime(LIB_OMP) < os.path.getmtime(SRC):
        try:
            _compile(LIB_OMP, ["-fopenmp"])
        except (subprocess.CalledProcessError, OSError):
            return None
    return LIB_OMP


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build_omp(force="--force" in sys.argv))
