"""Compile the fp64 CPU oracle (test infrastructure only).

Builds ``oracle/_build/<machine>/libkda_oracle.so`` from ``kda_oracle.c`` with gcc:
no fast-math, floating-point contraction off (identical bits on x86 and
Arm), OpenMP when the compiler supports it.
"""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
OUT_DIR = os.path.join(HERE, "_build", platform.machine())
LIB = os.path.join(OUT_DIR, "libkda_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
            "-shared", "-fPIC", SRC, "-o", LIB + ".tmp"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
