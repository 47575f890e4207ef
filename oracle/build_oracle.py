"""Compiles the C++ oracle (moe_oracle.cpp) into libmoe_oracle.so with g++.

Test infrastructure: building the checker does not run it.  Loaded on its own (no package import)
by the repository's build entry point, and used by moe_oracle.py to build the library on first use.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "libmoe_oracle.so")
# plain IEEE double arithmetic (no contraction into fused multiply-adds), portable x86-64 code (the
# library may be built on one host and run on another), OpenMP over independent rows
CXXFLAGS = ["-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-fvisibility=hidden",
            "-Wl,-Bsymbolic"]


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compiles the oracle library (when `out` is missing or older than `src`); returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(os.path.abspath(out)))
    os.close(fd)
    res = subprocess.run(["g++", *CXXFLAGS, "-o", tmp, src], capture_output=True, text=True)
    if res.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"g++ failed on {src}:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
