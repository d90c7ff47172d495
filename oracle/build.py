"""Build the CPU oracle shared library (plain g++, no CUDA).

TEST INFRASTRUCTURE ONLY: the oracle is never part of the product path.
``build()`` writes ``oracle/_build/libhs_oracle.so``; ``build(mutant=k)``
writes a copy with one deliberately planted mistake (``HSO_MUTANT=k``) that
the pin tests use to show that the pins catch it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
SRC = os.path.join(HERE, "hs_oracle.cpp")
HDR = os.path.join(HERE, "hs_oracle.h")


def lib_path(mutant: int = 0) -> str:
    name = "libhs_oracle.so" if mutant == 0 else f"libhs_oracle_mutant{mutant}.so"
    return os.path.join(BUILD_DIR, name)


def build(mutant: int = 0, force: bool = False) -> str:
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(SRC), os.path.getmtime(HDR))):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           f"-DHSO_MUTANT={int(mutant)}", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))
