"""Compile the C++ oracle into ``oracle/libparef.so`` (plain g++, no GPU).

Test infrastructure: the GPU library neither links nor loads this output.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "paref.cpp")
HDR = os.path.join(HERE, "paref.h")
LIB = os.path.join(HERE, "libparef.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-Wall", "-Wextra",
               SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
