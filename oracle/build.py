"""Build the C++ FP64 oracle (oracle/moe_oracle.cpp) into oracle/_lib/liboracle.so.

Test infrastructure only: plain g++ with OpenMP, no CUDA, nothing shared with
the CUDA library.  ``python -m oracle.build`` or ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "liboracle.so")

# -ffp-contract=off: no fused multiply-adds, so every fp32 decision of the
# quantisers is the IEEE result on any host (x86-64 or aarch64)
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def lib_path() -> str:
    return LIB


def build() -> str:
    cxx = os.environ.get("CXX") or shutil.which("g++") or "g++"
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx, *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build())
