"""CPU oracle for NF4 weight-quantized projections -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs import this package.  The product (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

This module is argument marshalling over ``nf4_oracle.c`` (plain C, float64
accumulation).  Arrays are numpy: weights fp32 ``[M, K]``, codes uint8
``[M, K/2]`` (low nibble = even k), scales fp32 ``[M, K/64]``, activations either
fp32 or bf16 bit patterns stored as uint16.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, library_path

F32 = 0
BF16 = 1

_lib = None


def load():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    src = os.path.join(os.path.dirname(__file__), "nf4_oracle.c")
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(src):
        build_oracle()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.nf4o_codebook.argtypes = [P]
    lib.nf4o_quantize.argtypes = [P, I64, I64, P, P]
    lib.nf4o_dequant.argtypes = [P, P, I64, I64, P]
    lib.nf4o_gemv.argtypes = [P, P, I64, I64, P, I, P, I64, P, P]
    lib.nf4o_gemv_residual.argtypes = [P, P, I64, I64, P, I, P, P, I64, P, P]
    lib.nf4o_gemv_swiglu.argtypes = [P, P, P, P, I64, I64, P, I, P, I64, P, P, P, P]
    lib.nf4o_gemv_argmax.argtypes = [P, P, I64, I64, P, I, P, P, P]
    lib.nf4o_gemm_chunk.argtypes = [P, P, I64, I64, P, I64, P, I64, P, P]
    lib.nf4o_gemv_qkv.argtypes = [P, P, P, P, I64, P, I, P, I64, P, P]
    lib.nf4o_dequant_rows.argtypes = [P, P, I64, I64, P, I64, P, P, P]
    lib.nf4o_gemv_glu_interleaved.argtypes = [P, P, I64, I64, P, I, P, I64, P, P, P, P]
    lib.nf4o_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_double, P, P]
    lib.nf4o_rmsnorm.restype = ctypes.c_int
    lib.nf4o_round_bf16.argtypes = [ctypes.c_double]
    lib.nf4o_round_bf16.restype = ctypes.c_uint16
    for name in ("nf4o_codebook", "nf4o_quantize", "nf4o_dequant", "nf4o_gemv", "nf4o_gemv_residual",
                 "nf4o_gemv_swiglu", "nf4o_gemv_argmax", "nf4o_gemm_chunk"):
        getattr(lib, name).restype = ctypes.c_int
    # the library's calls on the host (nf4_ref_*), weight descriptors by pointer
    W = ctypes.POINTER(RefWeight)
    ref = {"nf4_ref_quantize": [P, I64, I64, P, P], "nf4_ref_gemv": [W, P, I, P],
           "nf4_ref_gemv_residual": [W, P, I, P, P], "nf4_ref_gemv_swiglu": [W, W, P, I, P],
           "nf4_ref_gemv_glu_interleaved": [W, P, I, P], "nf4_ref_gemv_qkv": [W, W, W, P, P, P, P, I, P, P, P],
           "nf4_ref_gemv_argmax": [W, P, I, P, P], "nf4_ref_gemm_chunk": [W, P, I, P],
           "nf4_ref_dequant_rows": [W, P, I64, P, I], "nf4_ref_rmsnorm": [P, P, I64, I64, ctypes.c_float, P, I]}
    for name, args in ref.items():
        getattr(lib, name).argtypes = args
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


class RefWeight(ctypes.Structure):
    """Weight descriptor of the nf4_ref_* calls (host pointers): codes, scales, M, K."""

    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("K", ctypes.c_int64)]

    @classmethod
    def of(cls, codes: np.ndarray, scales: np.ndarray) -> "RefWeight":
        return cls(codes.ctypes.data, scales.ctypes.data, codes.shape[0], codes.shape[1] * 2)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(status, what):
    if status != 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {status})")


def _xtype(x):
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError("x must be float32 or uint16 (bf16 bits)")


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, len(r)


def codebook() -> np.ndarray:
    out = np.zeros(16, np.float32)
    load().nf4o_codebook(_ptr(out))
    return out


def quantize(W: np.ndarray):
    W = np.ascontiguousarray(W, dtype=np.float32)
    M, K = W.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 64), np.float32)
    _check(load().nf4o_quantize(_ptr(W), M, K, _ptr(codes), _ptr(scales)), "quantize")
    return codes, scales


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    M, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((M, K), np.float32)
    _check(load().nf4o_dequant(_ptr(codes), _ptr(scales), M, K, _ptr(out)), "dequant")
    return out


def gemv(codes, scales, x, rows=None):
    """float64 y and magnitude S for the requested rows (all rows if None)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    x = np.ascontiguousarray(x)
    M, K = codes.shape[0], codes.shape[1] * 2
    r, n = _rows(rows, M)
    y = np.zeros(n, np.float64)
    S = np.zeros(n, np.float64)
    _check(load().nf4o_gemv(_ptr(codes), _ptr(scales), M, K, _ptr(x), _xtype(x), _ptr(r), n, _ptr(y),
                            _ptr(S)), "gemv")
    return y, S


def gemv_residual(codes, scales, x, resid, rows=None):
    """(float64 y + r, fp32-rounded y + r) for the requested rows."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    x = np.ascontiguousarray(x)
    resid = np.ascontiguousarray(resid, np.float32)
    M, K = codes.shape[0], codes.shape[1] * 2
    r, n = _rows(rows, M)
    y64 = np.zeros(n, np.float64)
    y32 = np.zeros(n, np.float32)
    _check(load().nf4o_gemv_residual(_ptr(codes), _ptr(scales), M, K, _ptr(x), _xtype(x), _ptr(resid),
                                     _ptr(r), n, _ptr(y64), _ptr(y32)), "gemv_residual")
    return y64, y32


def gemv_qkv(parts, x, rows=None):
    """Fused q/k/v projection: parts = [(codes, scales, bias or None)] x 3 (q, k,
    v; same K).  float64 y and magnitude S over the concatenated row space (q
    rows, then k, then v), for the requested rows (all if None)."""
    assert len(parts) == 3
    cs = [np.ascontiguousarray(c, np.uint8) for c, _, _ in parts]
    ss = [np.ascontiguousarray(s_, np.float32) for _, s_, _ in parts]
    bs = [None if b is None else np.ascontiguousarray(b, np.float32) for _, _, b in parts]
    Ms = [c.shape[0] for c in cs]
    K = cs[0].shape[1] * 2
    assert all(c.shape[1] * 2 == K for c in cs)
    x = np.ascontiguousarray(x)
    r, n = _rows(rows, sum(Ms))
    V3 = ctypes.c_void_p * 3
    y = np.zeros(n, np.float64)
    S = np.zeros(n, np.float64)
    _check(load().nf4o_gemv_qkv(V3(*[_ptr(c) for c in cs]), V3(*[_ptr(s_) for s_ in ss]),
                                V3(*[_ptr(b) for b in bs]), (ctypes.c_int64 * 3)(*Ms), K, _ptr(x), _xtype(x),
                                _ptr(r), n, _ptr(y), _ptr(S)), "gemv_qkv")
    return y, S


def dequant_rows(codes, scales, ids):
    """Gathered, dequantized rows of an NF4 table: (fp32 [n, K], bf16 bits
    [n, K], number of ids outside the table, whose rows are zero)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    ids = np.ascontiguousarray(ids, np.int64)
    V, K = codes.shape[0], codes.shape[1] * 2
    n = ids.shape[0]
    f32 = np.zeros((n, K), np.float32)
    b16 = np.zeros((n, K), np.uint16)
    bad = np.zeros(1, np.int64)
    _check(load().nf4o_dequant_rows(_ptr(codes), _ptr(scales), V, K, _ptr(ids) if n else None, n, _ptr(f32),
                                    _ptr(b16), _ptr(bad)), "dequant_rows")
    return f32, b16, int(bad[0])


def gemv_swiglu(g_codes, g_scales, u_codes, u_scales, x, rows=None):
    """(float64 silu(g)*u, bf16 bits of it, float64 g, float64 u) for the rows."""
    args = [np.ascontiguousarray(a) for a in (g_codes, g_scales, u_codes, u_scales)]
    x = np.ascontiguousarray(x)
    M, K = args[0].shape[0], args[0].shape[1] * 2
    r, n = _rows(rows, M)
    o64 = np.zeros(n, np.float64)
    obf = np.zeros(n, np.uint16)
    g = np.zeros(n, np.float64)
    u = np.zeros(n, np.float64)
    _check(load().nf4o_gemv_swiglu(*[_ptr(a) for a in args], M, K, _ptr(x), _xtype(x), _ptr(r), n,
                                   _ptr(o64), _ptr(obf), _ptr(g), _ptr(u)), "gemv_swiglu")
    return o64, obf, g, u


def gemv_glu_interleaved(codes, scales, x, cols=None):
    """SwiGLU over one matrix whose rows alternate gate (even) and up (odd).

    Returns (float64 silu(g)*u, bf16 bits of it, float64 g, float64 u) for the
    outputs ``cols`` (all ``M2 / 2`` if None).
    """
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    x = np.ascontiguousarray(x)
    M2, K = codes.shape[0], codes.shape[1] * 2
    c, n = _rows(cols, M2 // 2)
    o64 = np.zeros(n, np.float64)
    obf = np.zeros(n, np.uint16)
    g = np.zeros(n, np.float64)
    u = np.zeros(n, np.float64)
    _check(load().nf4o_gemv_glu_interleaved(_ptr(codes), _ptr(scales), M2, K, _ptr(x), _xtype(x), _ptr(c), n,
                                            _ptr(o64), _ptr(obf), _ptr(g), _ptr(u)), "gemv_glu_interleaved")
    return o64, obf, g, u


def gemv_argmax(codes, scales, x):
    """(float64 logits, fp32 logits, argmax index with ties to the lowest)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    x = np.ascontiguousarray(x)
    M, K = codes.shape[0], codes.shape[1] * 2
    l64 = np.zeros(M, np.float64)
    l32 = np.zeros(M, np.float32)
    idx = np.zeros(1, np.int64)
    _check(load().nf4o_gemv_argmax(_ptr(codes), _ptr(scales), M, K, _ptr(x), _xtype(x), _ptr(l64),
                                   _ptr(l32), _ptr(idx)), "gemv_argmax")
    return l64, l32, int(idx[0])


def gemm_chunk(codes, scales, X_bf16, rows=None):
    """float64 Y [N, nrows] and magnitude S for the requested rows."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    X = np.ascontiguousarray(X_bf16, np.uint16)
    if X.ndim == 1:
        X = X[None, :]
    M, K = codes.shape[0], codes.shape[1] * 2
    N = X.shape[0]
    r, n = _rows(rows, M)
    Y = np.zeros((N, n), np.float64)
    S = np.zeros((N, n), np.float64)
    _check(load().nf4o_gemm_chunk(_ptr(codes), _ptr(scales), M, K, _ptr(X), N, _ptr(r), n, _ptr(Y),
                                  _ptr(S)), "gemm_chunk")
    return Y, S


def rmsnorm(x, w_bf16, eps):
    """RMSNorm of each row of x (fp32 [rows, K] or [K]) with bf16 gain bits
    w [K]: (float64 y, float64 mean squares).  "Decode V2 -- resident
    executor", section 3: x * rsqrt(mean(x^2) + eps) * w."""
    x = np.ascontiguousarray(x, np.float32)
    one = x.ndim == 1
    if one:
        x = x[None, :]
    w = np.ascontiguousarray(w_bf16, np.uint16)
    rows, K = x.shape
    if w.shape != (K,):
        raise ValueError("gain must have K elements")
    y = np.zeros((rows, K), np.float64)
    ms = np.zeros(rows, np.float64)
    _check(load().nf4o_rmsnorm(_ptr(x), _ptr(w), rows, K, float(eps), _ptr(y), _ptr(ms)), "rmsnorm")
    return (y[0], ms[0]) if one else (y, ms)


def round_bf16(v: float) -> int:
    """bf16 bits of v rounded to nearest even."""
    return int(load().nf4o_round_bf16(float(v)))
