"""The C ABI driven from plain C on the GPU (tests/c/abi_from_c.c): the program
quantizes a seeded 2048 x 11008 weight with nf4_quantize and runs
nf4_gemv_residual with bf16 x, through include/nf4.h and libnf4.so only, and
dumps its inputs and outputs.  The codes and scales must equal the oracle's
encoder bit for bit, and y must lie within the stated bound of the oracle's
float64 sum plus the residual.  (Named to run after the other GPU tests.)"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

from . import helpers as H

pytestmark = pytest.mark.gpu

M, K = 2048, 11008


def test_down_residual_from_c(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from .c.build_c import build_abi_program

    exe = build_abi_program(str(tmp_path))
    out = os.path.join(str(tmp_path), "dump.bin")
    r = subprocess.run([exe, out], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "device run ok" in r.stdout, r.stdout
    raw = open(out, "rb").read()
    sizes = [("W", np.float32, M * K), ("x", np.uint16, K), ("r", np.float32, M), ("codes", np.uint8, M * K // 2),
             ("scales", np.float32, M * K // 64), ("y", np.float32, M)]
    d, off = {}, 0
    for name, dt, n in sizes:
        nb = n * np.dtype(dt).itemsize
        d[name] = np.frombuffer(raw[off:off + nb], dtype=dt).copy()
        off += nb
    assert off == len(raw)
    W = d["W"].reshape(M, K)
    codes, scales = oracle.quantize(W)
    assert np.array_equal(d["codes"].reshape(M, K // 2), codes)
    assert np.array_equal(d["scales"].reshape(M, K // 64).view(np.uint32), scales.view(np.uint32))
    y64, _ = oracle.gemv_residual(codes, scales, d["x"], d["r"])
    _, S = oracle.gemv(codes, scales, d["x"])
    H.assert_within(d["y"], y64, S, extra=H.ulp_f32(y64), what="down + residual from C")
