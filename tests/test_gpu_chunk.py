"""GPU parity of the prefill chunk (nf4_gemm_chunk, tcgen05) against the oracle.

The oracle computes Y[n][m] = sum_k bf16(W_hat[m][k]) * X[n][k] in float64;
the kernel rounds the dequantized weights to bf16 the same way and accumulates
in fp32 on the tensor cores, so the stated bound 2e-3 * S (S over X[n]) holds
with a wide margin.  Cases span ragged row tiles (M not a multiple of 128),
every token count the survey lists (1, 7, 8, 16, 31, 32), the split-K path of
the full 14B shape (sampled rows), determinism and the workspace contract.
"""
from __future__ import annotations

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


def _run(nf4, codes, scales, X, ws=None):
    W = H.weight_tensors(codes, scales)
    Xt = H.bf16_tensor(X.reshape(-1)).view(X.shape[0], X.shape[1])
    M = codes.shape[0]
    Y = torch.full((X.shape[0] * M + 64,), 777.0, device="cuda")
    if ws is None:
        ws = nf4.new_workspace(M, codes.shape[1] * 2, X.shape[0])
    nf4.nf4_gemm_chunk(W, Xt, Y[:X.shape[0] * M].view(X.shape[0], M), workspace=ws)
    Yh = Y.cpu().numpy()
    assert np.all(Yh[X.shape[0] * M:] == 777.0), "wrote past Y"
    return Yh[:X.shape[0] * M].reshape(X.shape[0], M), ws


def _check(Y, codes, scales, X, rows=None, what=""):
    Yr, S = oracle.gemm_chunk(codes, scales, X, rows=rows)
    got = Y if rows is None else Y[:, rows]
    for n in range(X.shape[0]):
        H.assert_within(got[n], Yr[n], S[n], what=f"{what} n={n}")
    return float(np.max(np.abs(got - Yr) / np.maximum(S, 1e-300)))


@pytest.mark.parametrize("M,K,N", [(128, 64, 1), (128, 64, 32), (130, 128, 7), (256, 512, 16), (1000, 1024, 31),
                                   (300, 2048, 8), (64, 5120, 32), (2500, 256, 32)])
def test_chunk_shapes(nf4, M, K, N):
    seed = 500 + M + N
    codes, scales = H.quantized(seed, 0, M, K)
    X = synth.normal_bf16(seed, 1, N * K).reshape(N, K)
    Y, ws = _run(nf4, codes, scales, X)
    rel = _check(Y, codes, scales, X, what=f"chunk {M}x{K} N={N}")
    assert rel < 1e-5


@pytest.mark.parametrize("N", [1, 7, 8, 16, 31, 32])
def test_chunk_token_counts_split_k(nf4, N):
    # 14B-shaped rows but fewer of them: still split along K
    M, K = 1536, 5120
    codes, scales = H.quantized(600 + N, 0, M, K)
    X = synth.normal_bf16(600 + N, 1, N * K).reshape(N, K)
    Y, ws = _run(nf4, codes, scales, X)
    _check(Y, codes, scales, X, what=f"N={N}")
    # the tickets at the end of the workspace are left at zero
    nb = nf4.nf4_workspace_bytes(M, K, N)
    tail = ws[: nb].view(torch.uint8)[-((M + 127) // 128) * 4 - 16:]
    assert torch.count_nonzero(tail).item() == 0


def test_chunk_full_14b_sampled_rows_and_determinism(nf4):
    w = synth.WORKLOADS["chunk14b"]
    d = synth.workload_inputs(w)
    codes, scales = oracle.quantize(d["W"])
    Y1, ws = _run(nf4, codes, scales, d["X"])
    Y2, _ = _run(nf4, codes, scales, d["X"], ws)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32)), "chunk is not deterministic"
    g = np.random.Generator(np.random.PCG64(7))
    rows = np.unique(np.concatenate([np.arange(0, 13824, 97), [0, 127, 128, 13823], g.integers(0, 13824, 64)]))
    _check(Y1, codes, scales, d["X"], rows=rows, what="14B chunk")


def test_chunk_columns_match_gemv(nf4):
    M, K, N = 640, 2048, 5
    codes, scales = H.quantized(610, 0, M, K)
    X = synth.normal_bf16(610, 1, N * K).reshape(N, K)
    Y, _ = _run(nf4, codes, scales, X)
    W = H.weight_tensors(codes, scales)
    for n in range(N):
        y = nf4.nf4_gemv(W, H.bf16_tensor(X[n])).cpu().numpy().astype(np.float64)
        _, S = oracle.gemv(codes, scales, X[n])
        # both are within the stated bound of their own definitions; bf16 weight
        # rounding (<= 2^-9 relative) separates them
        assert np.all(np.abs(Y[n] - y) <= (2.0 ** -9 + 2e-3) * S)


def test_chunk_zero_level_rows(nf4):
    M, K, N = 200, 512, 4
    codes = np.full((M, K // 2), 0x77, np.uint8)
    scales = np.full((M, K // 64), 3.5, np.float32)
    X = synth.normal_bf16(620, 1, N * K).reshape(N, K)
    Y, _ = _run(nf4, codes, scales, X)
    assert np.all(Y == 0.0)


def test_chunk_kernel_choice_is_described(nf4):
    # K % 256 == 0: the stream-K TMA kernel (whole tiles per block when there are
    # at least four tiles per block); other K: the register-fed kernel
    assert "stream-K" in nf4.nf4_describe_config(13824, 5120, 32)
    assert "whole tiles per block" in nf4.nf4_describe_config(81920, 256, 5)
    assert "stream-K" not in nf4.nf4_describe_config(1000, 192, 4)


def test_chunk_whole_tiles_per_block(nf4):
    # 640 row tiles on 152 blocks: no tile is split, no partials
    M, K, N = 81920 + 40, 256, 5
    codes, scales = H.quantized(630, 0, M, K)
    X = synth.normal_bf16(630, 1, N * K).reshape(N, K)
    Y, _ = _run(nf4, codes, scales, X)
    _check(Y, codes, scales, X, what="whole tiles")


@pytest.mark.parametrize("M,K,N", [(384, 256, 32), (129, 768, 3), (1536, 2816, 17)])
def test_chunk_stream_k_ragged(nf4, M, K, N):
    # units of 256 columns split unevenly over the blocks, ragged last tile
    codes, scales = H.quantized(640 + M, 0, M, K)
    X = synth.normal_bf16(640 + M, 1, N * K).reshape(N, K)
    Y, ws = _run(nf4, codes, scales, X)
    _check(Y, codes, scales, X, what=f"stream-K {M}x{K} N={N}")
    Y2, _ = _run(nf4, codes, scales, X, ws)
    assert np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))


def test_chunk_fallback_kernel_unaligned_scales(nf4):
    # K % 256 == 0 but scales only 4-byte aligned: the register-fed kernel
    # (P-way split-K) runs instead of the TMA one; same definition, same bound
    M, K, N = 1000, 1024, 13
    codes, scales = H.quantized(650, 0, M, K)
    W = H.weight_tensors(codes, scales)
    buf = torch.zeros(scales.size + 4, dtype=torch.float32, device="cuda")
    buf[1:1 + scales.size].copy_(torch.from_numpy(scales.reshape(-1)))
    Wu = nf4.NF4Weight(W.codes, buf[1:1 + scales.size].view(M, K // 64))
    assert Wu.scales.data_ptr() % 16 == 4
    X = synth.normal_bf16(650, 1, N * K).reshape(N, K)
    Xt = H.bf16_tensor(X.reshape(-1)).view(N, K)
    ws = nf4.new_workspace(M, K, N)
    Y = torch.full((N, M), 777.0, device="cuda")
    nf4.nf4_gemm_chunk(Wu, Xt, Y, workspace=ws)
    _check(Y.cpu().numpy(), codes, scales, X, what="fallback chunk")
    Y2 = torch.full((N, M), 777.0, device="cuda")
    nf4.nf4_gemm_chunk(W, Xt, Y2, workspace=ws)  # aligned: the TMA kernel, same workspace
    _check(Y2.cpu().numpy(), codes, scales, X, what="TMA chunk after fallback")
    nb = nf4.nf4_workspace_bytes(M, K, N)
    tail = ws[:nb].view(torch.uint8)[-((M + 127) // 128) * 4 - 16:]
    assert torch.count_nonzero(tail).item() == 0
