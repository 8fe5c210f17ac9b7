"""Builds the float32 C++ oracle (``fp32_decoder.cpp``) into ``liboracle_fp32.so``.

Test infrastructure: plain g++ with no fused multiply-add
(``-ffp-contract=off``) and no fast-math, so every float operation of the
oracle is one IEEE single-precision operation in the order its source
writes it, on x86-64 and on aarch64 alike.  No CUDA, nothing shared with
the product library.
"""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp32_decoder.cpp")
LIB = os.path.join(HERE, "liboracle_fp32.so")
FLAGS = ["-O3", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math",
         "-fno-math-errno", "-Wall", "-Wextra"]


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(__file__))


def build(force: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("g++ is required to build the C++ oracle")
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([cxx, *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"g++ failed on the oracle:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv))
