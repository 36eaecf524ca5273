"""Builds liboracle.so from fab_oracle.cpp with the host C++ compiler.

TEST INFRASTRUCTURE ONLY: the oracle is the checker, never the product path.
Portable flags only (the same source builds on x86_64 and aarch64 hosts).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fab_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-O3", "-std=c++17", "-fPIC", "-shared", "-pthread", SRC, "-o", tmp]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
