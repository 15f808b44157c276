"""Compile the float64 C oracles (SSD scan, Mamba selective scan) into
``oracle/libssd_oracle.so``.

Test infrastructure: the oracle is what the CUDA library is checked against;
nothing in the product library uses it.  Portable C, no ISA flags, so the same
source builds on x86_64 and aarch64 hosts.  OpenMP is used when the compiler
has it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "ssd_oracle.c"), os.path.join(HERE, "mamba_oracle.c")]
LIB = os.path.join(HERE, "libssd_oracle.so")


def build_oracle(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in SRCS)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math"] + SRCS + ["-o", LIB, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
