"""Build the CPU oracle shared library (test infrastructure only).

Plain g++, no vectorisation flags that could change floating-point results:
-ffp-contract=off keeps a*b+c as two roundings on every host (GCC contracts to
FMA by default on aarch64), -fno-fast-math keeps IEEE semantics.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dkv_oracle.cpp")
LIB_PATH = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "dkv_oracle.h"))):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_oracle(force=True))
