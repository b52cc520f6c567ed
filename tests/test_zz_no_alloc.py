"""GPU test of nf4_gemm_chunk_noalloc, the prefill chunk for callers that
cannot allocate device memory (a host program that owns every allocation, or
a loop that must not call cudaMalloc because it synchronizes the device).

It is called through the C ABI, on two calls in a row, and each output is
compared with the CPU oracle's Y and with nf4_gemm_chunk given a caller
workspace: within the tests' bound 2e-3 * sum_k |bf16(W_hat) * X| per output.
The shapes reach both kernels that can run through the static scratch: the
TMA stream-K kernel (K a multiple of 256) and the register-fed kernel
(1000 x 320, whose K is split five ways, with partials and tickets in the
scratch).  This file sorts last so that a run stopping at its first failure
has already run every other test; it also passes when run alone in a fresh
process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from nf4_weight_quantized_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nf4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


def _noalloc(nf4, W, Xt, Y):
    w = W.struct()
    return nf4.lib.nf4_gemm_chunk_noalloc(ctypes.byref(w), ctypes.c_void_p(Xt.data_ptr()), Xt.shape[0],
                                          ctypes.c_void_p(Y.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,K,N", [(1536, 5120, 32), (1000, 1024, 7), (300, 2048, 1), (1000, 320, 7)])
def test_noalloc_matches_oracle_and_workspace_entry_point(nf4, M, K, N):
    seed = 900 + M + N
    codes, scales = H.quantized(seed, 0, M, K)
    X = synth.normal_bf16(seed, 1, N * K).reshape(N, K)
    Y_ref, S = oracle.gemm_chunk(codes, scales, X)
    W = H.weight_tensors(codes, scales)
    Xt = H.bf16_tensor(X.reshape(-1)).view(N, K)
    ref = nf4.nf4_gemm_chunk(W, Xt).cpu().numpy().astype(np.float64)
    for call in range(2):
        Y = torch.full((N, M), float("nan"), device="cuda")
        assert _noalloc(nf4, W, Xt, Y) == 0, nf4.nf4_last_error()
        got = Y.cpu().numpy().astype(np.float64)
        for n in range(N):
            H.assert_within(got[n], Y_ref[n], S[n], what=f"noalloc vs oracle, call {call} n={n}")
            H.assert_within(got[n], ref[n], S[n], what=f"noalloc vs nf4_gemm_chunk, call {call} n={n}")
    nf4.nf4_check_device_errors()


def test_noalloc_rejects_shapes_beyond_its_scratch(nf4):
    M, K, N = 65536, 5120, 32
    assert nf4.nf4_workspace_bytes(M, K, N) > 8 << 20
    W = nf4.NF4Weight(torch.zeros((M, K // 2), dtype=torch.uint8, device="cuda"),
                      torch.zeros((M, K // 64), dtype=torch.float32, device="cuda"))
    Xt = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((N, M), 5.0, device="cuda")
    assert _noalloc(nf4, W, Xt, Y) == -1
    assert "scratch" in nf4.nf4_last_error()
    torch.cuda.synchronize()
    assert torch.all(Y == 5.0).item(), "a rejected call must launch nothing"
