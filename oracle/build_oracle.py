"""Builds the C++ oracle (ia_oracle.cpp) into oracle/_build/libia_oracle.so.

Plain g++ (C++17, -O2, threads), with floating-point contraction off so that
every float32 and float64 operation is rounded on its own as IEEE 754
prescribes: the quantiser's decisions are defined by those roundings. The
library is test infrastructure (see ia_oracle.cpp); nothing in the CUDA
library uses it.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ia_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libia_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
         "-fno-fast-math", "-Wall"]


def up_to_date() -> bool:
    return os.path.exists(LIB) and all(os.path.getmtime(p) <= os.path.getmtime(LIB)
                                       for p in (SRC, __file__))


def build(force: bool = False) -> str:
    """Compile the oracle if its source changed; returns the library path."""
    if not force and up_to_date():
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("g++ not found: the C++ oracle cannot be built")
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([cxx] + FLAGS + [SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the oracle failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)  # atomic: concurrent builders leave one complete library
    return LIB


if __name__ == "__main__":
    print(build(force=True))
