"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol include/nf4.h declares, its codebook equals the oracle's bit for bit
(two independent derivations of the same closed form), and argument
validation fails before any device work."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf4.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:nf4_status|size_t|void|const char\*)\s+(nf4_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def nf4():
    from nf4_weight_quantized_gb300 import build

    if not os.path.exists(build.library_path()):
        build.build()
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("nf4_gemv", "nf4_gemv_residual", "nf4_gemv_swiglu", "nf4_gemv_argmax", "nf4_gemm_chunk",
              "nf4_workspace_bytes", "nf4_last_error", "nf4_describe_config"):
        assert n in names


def test_library_exports_every_declared_symbol(nf4):
    from nf4_weight_quantized_gb300 import build

    path = build.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW] (nf4_\w+)$", out, re.M))
    for name in _declared():
        assert name in exported, name
        assert getattr(nf4.lib, name) is not None
    assert set(nf4.EXPORTS) == set(_declared())


def test_library_codebook_equals_oracle(nf4, cb):
    lib_cb = np.array(nf4.nf4_codebook(), np.float32)
    assert np.array_equal(lib_cb.view(np.uint32), cb.view(np.uint32))


def test_workspace_bytes(nf4):
    assert nf4.nf4_workspace_bytes(151936, 2048, 1) == 16
    assert nf4.nf4_workspace_bytes(100, 65, 1) == 0
    assert nf4.nf4_workspace_bytes(100, 64, 0) == 0
    assert nf4.nf4_workspace_bytes(100, 64, 33) == 0


def test_validation_before_launch(nf4):
    lib = nf4.lib
    P = ctypes.c_void_p
    good = nf4.nf4_weight(4096, 4096, 8, 128)
    st = lib.nf4_gemv(ctypes.byref(nf4.nf4_weight(4096, 4096, 8, 100)), P(4096), 0, P(4096), None)
    assert st == -1 and "multiple of 64" in nf4.nf4_last_error()
    st = lib.nf4_gemv(ctypes.byref(nf4.nf4_weight(4096, 4096, 0, 128)), P(4096), 0, P(4096), None)
    assert st == -1
    st = lib.nf4_gemv(ctypes.byref(nf4.nf4_weight(4096, 4096, 8, 65536 + 64)), P(4096), 0, P(4096), None)
    assert st == -1
    st = lib.nf4_gemv(ctypes.byref(nf4.nf4_weight(4104, 4096, 8, 128)), P(4096), 0, P(4096), None)
    assert st == -2 and "codes" in nf4.nf4_last_error()
    st = lib.nf4_gemv(ctypes.byref(good), P(4100), 1, P(4096), None)
    assert st == -2 and "x" in nf4.nf4_last_error()
    st = lib.nf4_gemv(ctypes.byref(good), None, 1, P(4096), None)
    assert st == -3
    st = lib.nf4_gemv(ctypes.byref(good), P(4096), 7, P(4096), None)
    assert st == -1
    st = lib.nf4_gemv(None, P(4096), 0, P(4096), None)
    assert st == -3
    st = lib.nf4_gemv_swiglu(ctypes.byref(good), ctypes.byref(nf4.nf4_weight(4096, 4096, 9, 128)), P(4096), 1,
                             P(4096), None)
    assert st == -1 and "gate" in nf4.nf4_last_error()
    st = lib.nf4_gemv_argmax(ctypes.byref(good), P(4096), 1, P(4096), P(4100), P(4096), None)
    assert st == -2 and "index" in nf4.nf4_last_error()
    st = lib.nf4_gemm_chunk(ctypes.byref(good), P(4096), 33, P(4096), P(4096), None)
    assert st == -1 and "N = 33" in nf4.nf4_last_error()
    st = lib.nf4_gemm_chunk(ctypes.byref(good), P(4096), 0, P(4096), P(4096), None)
    assert st == -1
    st = lib.nf4_quantize(P(4096), 8, 96, P(4096), P(4096), None)
    assert st == -1


def test_no_device_is_reported_not_faked(nf4):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    good = nf4.nf4_weight(4096, 4096, 8, 128)
    st = nf4.lib.nf4_gemv(ctypes.byref(good), ctypes.c_void_p(4096), 0, ctypes.c_void_p(4096), None)
    assert st == -4  # NF4_ECUDA: no device, nothing launched, no fallback


def test_describe_config_rejects_bad_shape(nf4):
    assert "invalid shape" in nf4.nf4_describe_config(8, 100, 1)
    assert "invalid operation" in nf4.nf4_describe_launch("transpose", 8, 128, 1)
    assert "invalid operation" in nf4.nf4_describe_launch("residual", 8, 128, 4)  # N > 1 is the chunk only
    assert "invalid shape" in nf4.nf4_describe_launch("residual", 8, 100, 1)


def test_noalloc_rejects_oversize_before_any_device_work(nf4):
    # the scratch bound is checked on the host, before the device is touched
    big = nf4.nf4_weight(4096, 4096, 65536, 5120)
    st = nf4.lib.nf4_gemm_chunk_noalloc(ctypes.byref(big), ctypes.c_void_p(4096), 32, ctypes.c_void_p(4096), None)
    assert st == -1 and "scratch" in nf4.nf4_last_error()
    st = nf4.lib.nf4_gemm_chunk_noalloc(ctypes.byref(nf4.nf4_weight(4096, 4096, 8, 100)), ctypes.c_void_p(4096), 4,
                                        ctypes.c_void_p(4096), None)
    assert st == -1 and "multiple of 64" in nf4.nf4_last_error()


def test_c_program_uses_the_abi_without_python(tmp_path):
    # a plain C caller: codebook, argument checks and workspace sizes through
    # include/nf4.h and libnf4.so alone (no device needed)
    from .c.build_c import build_abi_program

    exe = build_abi_program(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "host checks ok" in r.stdout
