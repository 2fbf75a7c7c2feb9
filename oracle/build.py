"""Builds libmoe_oracle.so, the C++ CPU oracle, in-tree with g++.

TEST INFRASTRUCTURE: the library is the checker of the CUDA path, loaded only
by tests/, __graft_entry__.smoke() and bench.py's CPU legs.

    python -m oracle.build [--force]

Flags: -O2 and no fast-math; -ffp-contract=off keeps every multiply and add
a separately rounded IEEE operation, as the source writes them.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
HDR = os.path.join(HERE, "moe_oracle.h")
LIB = os.path.join(HERE, "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math",
         "-Wall", "-Wextra"]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR))


def build(force: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    cxx = shutil.which("g++") or "g++"
    tmp = LIB + ".tmp"
    subprocess.run([cxx] + FLAGS + ["-o", tmp, SRC], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    print(build(ap.parse_args().force))
