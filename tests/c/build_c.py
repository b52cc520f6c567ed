"""Compile tests/c/abi_from_c.c against include/nf4.h, libnf4.so and the CUDA
runtime with the host C compiler (test infrastructure)."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))


def cuda_dirs():
    """(include dir, directory holding libcudart.so) of the CUDA toolkit."""
    base = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libs = [os.path.join(base, "lib64")] + sorted(glob.glob(os.path.join(base, "targets", "*", "lib")))
    lib = next((d for d in libs if glob.glob(os.path.join(d, "libcudart.so*"))), libs[0])
    return os.path.join(base, "include"), lib


def build_abi_program(out_dir: str) -> str:
    from nf4_weight_quantized_gb300 import build

    if not os.path.exists(build.library_path()):
        build.build()
    libdir = os.path.dirname(build.library_path())
    inc, cudalib = cuda_dirs()
    exe = os.path.join(out_dir, "abi_from_c")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"), "-I", inc,
           os.path.join(HERE, "abi_from_c.c"), "-o", exe, "-L", libdir, "-lnf4", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe
