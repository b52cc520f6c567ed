"""Shared helpers for the GPU parity tests: seeded inputs, oracle references and
the tolerance checks.  Tolerances (the stated bound of the method):

* fp32 outputs:  |y - y_ref| <= 2e-3 * S_m,  S_m = sum_k |x_k * W_hat[m][k]|
* residual:      the same plus one fp32 ulp of |y_ref| (the final add rounds)
* bf16 SwiGLU:   the fp32 bound on g and u propagated through silu(g) * u
                 (|silu'| <= 1.1) plus one bf16 ulp of |out_ref|
* argmax index:  bit-exact, ties to the lowest index
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from nf4_weight_quantized_gb300 import synth

EPS = 2e-3


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).to(device).view(torch.bfloat16)


def x_tensor(x: np.ndarray, device="cuda") -> torch.Tensor:
    if x.dtype == np.uint16:
        return bf16_tensor(x, device)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def bf16_bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def weight_tensors(codes: np.ndarray, scales: np.ndarray, device="cuda"):
    from nf4_weight_quantized_gb300 import nf4

    return nf4.NF4Weight(torch.from_numpy(np.ascontiguousarray(codes)).to(device),
                         torch.from_numpy(np.ascontiguousarray(scales)).to(device))


def make_x(seed: int, K: int, dtype: str) -> np.ndarray:
    return synth.normal_f32(seed, 1, K) if dtype == "f32" else synth.normal_bf16(seed, 1, K)


def quantized(seed: int, tid: int, M: int, K: int):
    return oracle.quantize(synth.weights(seed, tid, M, K))


def assert_within(gpu, ref, S, extra=0.0, what=""):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    bound = EPS * S + extra
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {len(ref)} outside the bound; first rows {bad[:5]}, "
                           f"err {err[bad[:5]]}, bound {bound[bad[:5]]}")
    return float(np.max(err / np.maximum(S, 1e-300))) if len(S) else 0.0


def ulp_f32(v):
    return np.spacing(np.abs(np.asarray(v, np.float32))).astype(np.float64)


def ulp_bf16(v):
    a = np.abs(np.asarray(v, np.float64))
    out = np.empty_like(a)
    nz = a >= 2.0 ** -126
    out[nz] = 2.0 ** (np.floor(np.log2(a[nz])) - 7)
    out[~nz] = 2.0 ** -133
    return out


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_bound(g, u, Sg, Su):
    tg, tu = EPS * Sg, EPS * Su
    return 1.1 * tg * (np.abs(u) + tu) + (np.abs(silu(g)) + 1.1 * tg) * tu


def top2_gap(y: np.ndarray):
    """Gap between the two largest DISTINCT values (rows that tie exactly are
    one value: their order is fixed by the lowest-index rule)."""
    u = np.unique(np.asarray(y, np.float64))
    return float(u[-1] - u[-2]) if len(u) > 1 else math.inf
