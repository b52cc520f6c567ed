"""Python binding of libnf4 (ctypes).  Argument marshalling only.

Every function here takes torch CUDA tensors, checks dtypes/devices/shapes,
and calls the C entry point of the same name in ``libnf4.so`` on the current
(or given) CUDA stream.  All arithmetic runs in the library's kernels; there is
no fallback.  Importing this module fails loudly if the library is not built.

Output tensors are allocated with torch when the caller does not pass them;
callers that need an allocation-free step (CUDA-graph capture, an arena)
pass every output and workspace explicitly.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from .build import library_path

NF4_F32 = 0
NF4_BF16 = 1
MAX_K = 65536
MAX_CHUNK_N = 32

_STATUS = {0: "NF4_OK", -1: "NF4_EINVAL", -2: "NF4_EALIGN", -3: "NF4_ENULL", -4: "NF4_ECUDA", -5: "NF4_EARCH",
           -6: "NF4_ETIMEOUT", -7: "NF4_ERANGE"}


class NF4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class nf4_weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("K", ctypes.c_int64)]


def _load():
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"libnf4.so is not built ({path} missing): run __graft_entry__.build() "
                          "or python nf4_weight_quantized_gb300/build.py")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    W = ctypes.POINTER(nf4_weight)
    sig = {
        "nf4_gemv": [W, P, I, P, P],
        "nf4_gemv_residual": [W, P, I, P, P, P],
        "nf4_gemv_swiglu": [W, W, P, I, P, P],
        "nf4_gemv_glu_interleaved": [W, P, I, P, P],
        "nf4_gemv_qkv": [W, W, W, P, P, P, P, I, P, P, P, P],
        "nf4_dequant_rows": [W, P, ctypes.c_int64, P, I, P],
        "nf4_gemv_argmax": [W, P, I, P, P, P, P],
        "nf4_gemm_chunk": [W, P, I, P, P, P],
        "nf4_gemm_chunk_noalloc": [W, P, I, P, P],
        "nf4_quantize": [P, ctypes.c_int64, ctypes.c_int64, P, P, P],
        "nf4_rmsnorm": [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, P, I, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.nf4_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.nf4_workspace_bytes.restype = ctypes.c_size_t
    lib.nf4_codebook.argtypes = [P]
    lib.nf4_codebook.restype = None
    lib.nf4_last_error.argtypes = []
    lib.nf4_last_error.restype = ctypes.c_char_p
    lib.nf4_describe_config.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.nf4_describe_config.restype = ctypes.c_char_p
    lib.nf4_describe_launch.argtypes = [ctypes.c_char_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.nf4_describe_launch.restype = ctypes.c_char_p
    lib.nf4_check_device_errors.argtypes = []
    lib.nf4_check_device_errors.restype = ctypes.c_int
    lib.nf4_debug_set_wait_limit.argtypes = [ctypes.c_uint32]
    lib.nf4_debug_set_wait_limit.restype = None
    return lib


lib = _load()

EXPORTS = ("nf4_gemv", "nf4_gemv_residual", "nf4_gemv_swiglu", "nf4_gemv_argmax", "nf4_gemm_chunk",
           "nf4_workspace_bytes", "nf4_quantize", "nf4_codebook", "nf4_last_error", "nf4_describe_config",
           "nf4_describe_launch", "nf4_check_device_errors", "nf4_gemm_chunk_noalloc", "nf4_gemv_qkv",
           "nf4_dequant_rows", "nf4_gemv_glu_interleaved", "nf4_debug_set_wait_limit", "nf4_rmsnorm")


def _check(status: int):
    if status != 0:
        raise NF4Error(status, lib.nf4_last_error().decode())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, numel=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def _xtype(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return NF4_F32
    if x.dtype == torch.bfloat16:
        return NF4_BF16
    raise TypeError("activations must be float32 or bfloat16")


@dataclass
class NF4Weight:
    """An NF4 matrix on the device: codes uint8 [M, K/2] and scales fp32 [M, K/64]."""

    codes: torch.Tensor
    scales: torch.Tensor

    @property
    def M(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] * 2

    def struct(self) -> nf4_weight:
        _dev(self.codes, "codes", torch.uint8)
        _dev(self.scales, "scales", torch.float32, self.M * (self.K // 64))
        return nf4_weight(self.codes.data_ptr(), self.scales.data_ptr(), self.M, self.K)


def nf4_quantize(W: torch.Tensor, codes: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                 stream=None) -> NF4Weight:
    M, K = W.shape
    if codes is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((M, max(K // 64, 1)), dtype=torch.float32, device=W.device)
    _check(lib.nf4_quantize(_dev(W, "W", torch.float32), M, K, _dev(codes, "codes", torch.uint8),
                            _dev(scales, "scales", torch.float32), _stream(stream)))
    return NF4Weight(codes, scales)


def nf4_gemv(W: NF4Weight, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if y is None:
        y = torch.empty(W.M, dtype=torch.float32, device=x.device)
    w = W.struct()
    _check(lib.nf4_gemv(ctypes.byref(w), _dev(x, "x", numel=W.K), _xtype(x), _dev(y, "y", torch.float32, W.M),
                        _stream(stream)))
    return y


def nf4_gemv_residual(W: NF4Weight, x: torch.Tensor, residual: torch.Tensor, y: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    if y is None:
        y = torch.empty(W.M, dtype=torch.float32, device=x.device)
    w = W.struct()
    _check(lib.nf4_gemv_residual(ctypes.byref(w), _dev(x, "x", numel=W.K), _xtype(x),
                                 _dev(residual, "residual", torch.float32, W.M),
                                 _dev(y, "y", torch.float32, W.M), _stream(stream)))
    return y


def nf4_gemv_swiglu(Wg: NF4Weight, Wu: NF4Weight, x: torch.Tensor, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(Wg.M, dtype=torch.bfloat16, device=x.device)
    g, u = Wg.struct(), Wu.struct()
    _check(lib.nf4_gemv_swiglu(ctypes.byref(g), ctypes.byref(u), _dev(x, "x", numel=Wg.K), _xtype(x),
                               _dev(out, "out", torch.bfloat16, Wg.M), _stream(stream)))
    return out


def nf4_gemv_glu_interleaved(W: NF4Weight, x: torch.Tensor, out: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """SwiGLU over one matrix whose rows alternate gate (even) and up (odd):
    out[c] = bf16(silu(v[2c]) * v[2c + 1]), v = W x; [W.M / 2] bf16."""
    if out is None:
        out = torch.empty(W.M // 2, dtype=torch.bfloat16, device=x.device)
    w = W.struct()
    _check(lib.nf4_gemv_glu_interleaved(ctypes.byref(w), _dev(x, "x", numel=W.K), _xtype(x),
                                        _dev(out, "out", torch.bfloat16, W.M // 2), _stream(stream)))
    return out


def nf4_gemv_qkv(Wq: NF4Weight, Wk: NF4Weight, Wv: NF4Weight, x: torch.Tensor, bq: torch.Tensor | None = None,
                 bk: torch.Tensor | None = None, bv: torch.Tensor | None = None, q: torch.Tensor | None = None,
                 k: torch.Tensor | None = None, v: torch.Tensor | None = None, stream=None):
    """One launch over the q, k and v rows sharing x, each bias (fp32, or None)
    added to its own rows.  Returns (q, k, v), fp32."""
    outs = []
    for o, W in ((q, Wq), (k, Wk), (v, Wv)):
        outs.append(torch.empty(W.M, dtype=torch.float32, device=x.device) if o is None else o)
    ws = [Wq.struct(), Wk.struct(), Wv.struct()]
    bias = [None if b is None else _dev(b, name, torch.float32, W.M)
            for b, name, W in ((bq, "bq", Wq), (bk, "bk", Wk), (bv, "bv", Wv))]
    _check(lib.nf4_gemv_qkv(ctypes.byref(ws[0]), ctypes.byref(ws[1]), ctypes.byref(ws[2]), *bias,
                            _dev(x, "x", numel=Wq.K), _xtype(x),
                            *[_dev(o, n, torch.float32, W.M) for o, n, W in zip(outs, "qkv", (Wq, Wk, Wv))],
                            _stream(stream)))
    return tuple(outs)


def nf4_dequant_rows(E: NF4Weight, ids: torch.Tensor, out: torch.Tensor | None = None,
                     dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """Rows E_hat[ids] of an NF4 table, [len(ids), K], fp32 (exact) or bf16."""
    n = ids.numel()
    if out is None:
        out = torch.empty((n, E.K), dtype=dtype, device=ids.device)
    ot = _xtype(out)
    e = E.struct()
    _check(lib.nf4_dequant_rows(ctypes.byref(e), _dev(ids, "ids", torch.int64, n) if n else None, n,
                                _dev(out, "out", out.dtype, n * E.K) if n else None, ot, _stream(stream)))
    return out


def nf4_rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float, out: torch.Tensor | None = None,
                dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """RMSNorm of each row of x (fp32 [K] or [rows, K]) with bf16 gain w [K]:
    x * w / sqrt(mean(x^2) + eps), fp32 or bf16; `out` may be x itself (fp32)."""
    if x.dim() not in (1, 2):
        raise ValueError("x must be [K] or [rows, K]")
    K = x.shape[-1]
    rows = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty(x.shape, dtype=dtype, device=x.device)
    _check(lib.nf4_rmsnorm(_dev(x, "x", torch.float32), _dev(w, "w", torch.bfloat16, K), rows, K, float(eps),
                           _dev(out, "out", out.dtype, rows * K), _xtype(out), _stream(stream)))
    return out


def nf4_workspace_bytes(M: int, K: int, N: int = 1) -> int:
    return int(lib.nf4_workspace_bytes(M, K, N))


def new_workspace(M: int, K: int, N: int = 1, device="cuda") -> torch.Tensor:
    """A zeroed workspace for nf4_gemv_argmax (N=1) or nf4_gemm_chunk (N>1)."""
    n = max(nf4_workspace_bytes(M, K, N), 16)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def nf4_gemv_argmax(W: NF4Weight, x: torch.Tensor, logits: torch.Tensor | None = None,
                    index: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None):
    if logits is None:
        logits = torch.empty(W.M, dtype=torch.float32, device=x.device)
    if index is None:
        index = torch.empty(1, dtype=torch.int64, device=x.device)
    if workspace is None:
        workspace = new_workspace(W.M, W.K, 1, x.device)
    w = W.struct()
    _check(lib.nf4_gemv_argmax(ctypes.byref(w), _dev(x, "x", numel=W.K), _xtype(x),
                               _dev(logits, "logits", torch.float32, W.M), _dev(index, "index", torch.int64, 1),
                               _dev(workspace, "workspace"), _stream(stream)))
    return logits, index


def nf4_gemm_chunk(W: NF4Weight, X: torch.Tensor, Y: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if X.dim() != 2 or X.shape[1] != W.K:
        raise ValueError("X must be [N, K]")
    N = X.shape[0]
    if Y is None:
        Y = torch.empty((N, W.M), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = new_workspace(W.M, W.K, N, X.device)
    w = W.struct()
    _check(lib.nf4_gemm_chunk(ctypes.byref(w), _dev(X, "X", torch.bfloat16), N,
                              _dev(Y, "Y", torch.float32, N * W.M), _dev(workspace, "workspace"),
                              _stream(stream)))
    return Y


def nf4_gemm_chunk_noalloc(W: NF4Weight, X: torch.Tensor, Y: torch.Tensor, stream=None) -> torch.Tensor:
    """nf4_gemm_chunk with the library's static scratch instead of a workspace.

    For callers that cannot allocate device memory; Y must be passed.  Calls
    that overlap on the GPU share the scratch and race."""
    if X.dim() != 2 or X.shape[1] != W.K:
        raise ValueError("X must be [N, K]")
    N = X.shape[0]
    w = W.struct()
    _check(lib.nf4_gemm_chunk_noalloc(ctypes.byref(w), _dev(X, "X", torch.bfloat16), N,
                                      _dev(Y, "Y", torch.float32, N * W.M), _stream(stream)))
    return Y


def nf4_codebook() -> list[float]:
    out = (ctypes.c_float * 16)()
    lib.nf4_codebook(ctypes.cast(out, ctypes.c_void_p))
    return list(out)


def nf4_describe_config(M: int, K: int, N: int = 1) -> str:
    return lib.nf4_describe_config(M, K, N).decode()


def nf4_describe_launch(op: str, M: int, K: int, N: int = 1) -> str:
    return lib.nf4_describe_launch(op.encode(), M, K, N).decode()


def nf4_check_device_errors() -> None:
    """Synchronize; raise NF4Error(NF4_ETIMEOUT) if a kernel's bounded wait ran out, or
    NF4Error(NF4_ERANGE) if nf4_dequant_rows met an id outside its table."""
    _check(lib.nf4_check_device_errors())


def nf4_debug_set_wait_limit(polls: int) -> None:
    """Failure-detection tests only: poll limit of the kernels' waits for staged
    weights (0 restores the default)."""
    lib.nf4_debug_set_wait_limit(int(polls))


def nf4_last_error() -> str:
    return lib.nf4_last_error().decode()
