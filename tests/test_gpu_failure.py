"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait of the bulk-copy GEMV and of the TMA prefill-chunk kernel on a
shared-memory barrier is bounded.  nf4_debug_set_wait_limit shortens the
pipeline waits (a producer's wait for a free stage, a consumer's wait for
staged weights or dequantized operands) to one non-blocking poll, on an
ordinary valid call whose copies all complete.  A producer that has filled its
ring always finds the next stage still in use at that poll (its consumers are
computing), so every block whose rows need more stages than its ring holds
gives up: it skips its outputs, waits (with the full limit) for the copies and
tensor-core work it issued, frees its tensor memory and sets the error word.  The tests check that
nf4_check_device_errors reports NF4_ETIMEOUT, that whatever the GEMV did write
is still correct, and that the next ordinary call in the same process is
correct and clean.  Nothing waits on a flag that is never set and nothing
faults.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nf4_weight_quantized_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu

NF4_ETIMEOUT = -6
SENTINEL = 12345.0


@pytest.fixture(scope="module")
def nf4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


def _timed_out(nf4, call):
    """Run `call` with one-poll waits; return the status nf4_check_device_errors gave."""
    nf4.nf4_check_device_errors()  # start clean
    nf4.nf4_debug_set_wait_limit(1)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        nf4.nf4_debug_set_wait_limit(0)
    try:
        nf4.nf4_check_device_errors()
    except nf4.NF4Error as e:
        return e.status
    return 0


def test_gemv_wait_runs_out_then_recovers(nf4):
    # 32768 rows of 2048: each block owns ~216 rows in several refills of its
    # stage ring, so its consumers wait on copies issued while they compute
    M, K = 32768, 2048
    codes, scales = H.quantized(960, 0, M, K)
    x = H.make_x(960, K, "bf16")
    y_ref, S = oracle.gemv(codes, scales, x)
    W = H.weight_tensors(codes, scales)
    xt = H.x_tensor(x)
    y = torch.full((M,), SENTINEL, device="cuda")
    status = _timed_out(nf4, lambda: nf4.nf4_gemv(W, xt, y))
    assert status == NF4_ETIMEOUT
    yh = y.cpu().numpy()
    written = yh != SENTINEL
    assert not np.all(written), "no block gave up"
    # rows a block finished before giving up are correct; the rest untouched
    H.assert_within(yh[written], y_ref[written], S[written], what="rows written before the timeout")
    # the library recovers: the same call with the default limit is correct
    y2 = nf4.nf4_gemv(W, xt).cpu().numpy()
    H.assert_within(y2, y_ref, S, what="gemv after a timeout")
    nf4.nf4_check_device_errors()


def test_chunk_wait_runs_out_then_recovers(nf4):
    # the 14B-shaped chunk: stream-K over 2160 units on persistent blocks, each
    # with tensor memory allocated; a timed-out block must still free it (the
    # next call allocates it again) and leave the workspace's tickets zeroed
    M, K, N = 13824, 5120, 32
    codes, scales = H.quantized(961, 0, M, K)
    X = synth.normal_bf16(961, 1, N * K).reshape(N, K)
    W = H.weight_tensors(codes, scales)
    Xt = H.bf16_tensor(X.reshape(-1)).view(N, K)
    ws = nf4.new_workspace(M, K, N)
    Y = torch.full((N, M), SENTINEL, device="cuda")
    status = _timed_out(nf4, lambda: nf4.nf4_gemm_chunk(W, Xt, Y, ws))
    assert status == NF4_ETIMEOUT
    nbytes = nf4.nf4_workspace_bytes(M, K, N)
    tickets = ws[nbytes - 16 - ((M + 127) // 128) * 4:nbytes]  # per-tile tickets, then 16 spare bytes
    assert torch.count_nonzero(tickets).item() == 0, "tickets not left zeroed"
    # recovery: sampled rows of a normal call against the oracle
    Y2 = nf4.nf4_gemm_chunk(W, Xt, workspace=ws).cpu().numpy().astype(np.float64)
    rows = np.unique(np.concatenate([np.arange(0, M, 997), [M - 1]]))
    Y_ref, SY = oracle.gemm_chunk(codes[rows], scales[rows], X)
    for n in range(N):
        H.assert_within(Y2[n, rows], Y_ref[n], SY[n], what=f"chunk after a timeout n={n}")
    nf4.nf4_check_device_errors()
