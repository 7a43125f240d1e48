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
# the sanitized variant (AddressSanitizer + UndefinedBehaviorSanitizer, every
# finding fatal), loaded when ORACLE_LIBRARY=sanitized
LIB_PATH_SAN = os.path.join(HERE, "liboracle_san.so")
SAN_FLAGS = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g"]


def build_oracle(force: bool = False, sanitize: bool = False) -> str:
    lib = LIB_PATH_SAN if sanitize else LIB_PATH
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "dkv_oracle.h"))):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O1" if sanitize else "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra", *(SAN_FLAGS if sanitize else []), "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_oracle(force=True))
