"""Compile the CPU oracle (plain C) into a shared library with gcc.

Test infrastructure: building the checker is not using it.  ``-ffp-contract=off``
keeps gcc from fusing multiply-adds, so x86_64 and aarch64 hosts compute the
same float64 sums.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libnf4_oracle.so")


def build_oracle() -> str:
    out = library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           os.path.join(_HERE, "nf4_oracle.c"), "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle())
