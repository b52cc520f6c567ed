"""GPU parity of nf4_gemv_glu_interleaved (SwiGLU over one matrix whose rows
alternate gate and up: "gizai:tensor/lazy", method Lazy.gluIn) against the
oracle, through the C ABI.

Each output must lie within the SwiGLU bound derived from the stated GEMV
tolerance (|v - v_ref| <= 2e-3 * sum_k |x_k W_hat[m][k]| on both rows of the
pair) plus one bf16 ulp.  Shapes cover every kernel branch (one warp per row,
two chunks per thread, one and two chunks per thread with cross-warp sums),
ragged row counts, the register-prefetch kernel, and the full 3B gate/up pair
interleaved into one 22016 x 2048 matrix.
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


def _interleaved(seed, n_out, K):
    """Codes and scales of 2 * n_out rows: row 2c gate c, row 2c + 1 up c."""
    W = np.empty((2 * n_out, K), np.float32)
    W[0::2] = synth.weights(seed, 0, n_out, K)
    W[1::2] = synth.weights(seed, 1, n_out, K)
    return oracle.quantize(W)


def _check(nf4, W, codes, scales, x, what):
    o64, ref_bits, g, u = oracle.gemv_glu_interleaved(codes, scales, x)
    _, S = oracle.gemv(codes, scales, x)
    out = nf4.nf4_gemv_glu_interleaved(W, H.x_tensor(x))
    assert out.shape == (codes.shape[0] // 2,) and out.dtype == torch.bfloat16
    ob = H.bf16_bits_of(out)
    of = synth.bf16_to_f32(ob).astype(np.float64)
    bound = H.swiglu_bound(g, u, S[0::2], S[1::2]) + H.ulp_bf16(o64)
    err = np.abs(of - o64)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, f"{what}: outputs {bad[:5]} err {err[bad[:5]]} bound {bound[bad[:5]]}"
    return ob, ref_bits


@pytest.mark.parametrize("n_out,K", [(1, 64), (45, 2048), (300, 5120), (70, 11008), (2500, 1024), (3, 32768)])
@pytest.mark.parametrize("xd", ["f32", "bf16"])
def test_glu_interleaved_shapes(nf4, n_out, K, xd):
    seed = 600 + n_out
    codes, scales = _interleaved(seed, n_out, K)
    x = H.make_x(seed, K, xd)
    _check(nf4, H.weight_tensors(codes, scales), codes, scales, x, f"glu {2 * n_out}x{K} {xd}")
    nf4.nf4_check_device_errors()


@pytest.mark.parametrize("n_out,K", [(150, 2048), (77, 5120)])
def test_glu_interleaved_register_kernel(nf4, n_out, K):
    # scales that are 4- but not 16-byte aligned take the register-prefetch kernel
    codes, scales = _interleaved(650 + n_out, n_out, K)
    W = H.weight_tensors(codes, scales)
    sc = torch.empty(scales.size + 4, dtype=torch.float32, device="cuda")
    sc[1:1 + scales.size] = W.scales.reshape(-1)
    W2 = nf4.NF4Weight(W.codes, sc[1:1 + scales.size].view(2 * n_out, K // 64))
    assert W2.scales.data_ptr() % 16 != 0
    _check(nf4, W2, codes, scales, H.make_x(650 + n_out, K, "bf16"), f"glu register {2 * n_out}x{K}")
    nf4.nf4_check_device_errors()


def test_glu_interleaved_matches_two_matrix_swiglu(nf4):
    # the same pairs through both layouts (one interleaved matrix, or the even
    # rows as gate and the odd rows as up): both within the oracle's bound
    n_out, K = 1000, 2048
    codes, scales = _interleaved(660, n_out, K)
    x = H.make_x(660, K, "bf16")
    _check(nf4, H.weight_tensors(codes, scales), codes, scales, x, "glu 2000x2048")
    o64, _, g, u = oracle.gemv_glu_interleaved(codes, scales, x)
    _, S = oracle.gemv(codes, scales, x)
    two = nf4.nf4_gemv_swiglu(H.weight_tensors(codes[0::2], scales[0::2]),
                              H.weight_tensors(codes[1::2], scales[1::2]), H.x_tensor(x))
    b = synth.bf16_to_f32(H.bf16_bits_of(two)).astype(np.float64)
    bound = H.swiglu_bound(g, u, S[0::2], S[1::2]) + H.ulp_bf16(o64)
    assert np.all(np.abs(b - o64) <= bound)


def test_glu_interleaved_full_3b_gate_up(nf4):
    # the 3B MLP's gate and up projections (11008 x 2048 each) as one
    # interleaved 22016 x 2048 matrix, every output compared
    w = synth.WORKLOADS["swiglu"]
    d = synth.workload_inputs(w)
    W = np.empty((2 * w.M, w.K), np.float32)
    W[0::2], W[1::2] = d["W"], d["Wu"]
    codes, scales = oracle.quantize(W)
    ob, ref_bits = _check(nf4, H.weight_tensors(codes, scales), codes, scales, d["x"], "glu full 3B")
    assert np.mean(ob == ref_bits) > 0.99  # fp32-accurate sums: nearly all round like the oracle


def test_glu_interleaved_errors(nf4):
    K = 128
    codes, scales = _interleaved(670, 4, K)
    W = H.weight_tensors(codes, scales)
    x = H.x_tensor(H.make_x(670, K, "f32"))
    odd = nf4.NF4Weight(W.codes[:7], W.scales[:7])
    with pytest.raises(nf4.NF4Error, match="NF4_EINVAL"):  # rows come in pairs
        nf4.nf4_gemv_glu_interleaved(odd, x, out=torch.empty(3, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):  # out must hold W.M / 2 values
        nf4.nf4_gemv_glu_interleaved(W, x, out=torch.empty(8, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(TypeError):
        nf4.nf4_gemv_glu_interleaved(W, x, out=torch.empty(4, dtype=torch.float32, device="cuda"))
