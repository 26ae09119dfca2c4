"""Compile the fp64 CPU oracle (plain C + OpenMP) into oracle/libmla_oracle.so.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg load it; the product library never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libmla_oracle.so")
SRC = os.path.join(HERE, "mla_oracle.c")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "mla_oracle.h")))):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    # -ffp-contract=off keeps every multiply and add a separate fp64 rounding.
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=HERE)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
