"""GPU parity of nf4_rmsnorm (RMSNorm as its own one-block-per-row kernel,
"Decode V2 -- resident executor", section 3) against the oracle, through the
C ABI.

Bound, per element, against the oracle's float64 value y_ref:
  fp32 out:  |y - y_ref| <= 256 * 2^-24 * |y_ref|
  bf16 out:  the same plus one bf16 ulp of |y_ref|
The fp32 sum of squares has at most ~100 sequential roundings (K / threads per
thread, five shuffle levels, at most 32 warp totals), which enter the result
at half weight through the square root; the mean, eps, square root, division
and the two products add six more.  256 ulps covers that with room, and stays
far below the effect of a misplaced eps (eps = 0.5 cases) or a wrong mean.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nf4_weight_quantized_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu

REL = 256 * 2.0 ** -24


@pytest.fixture(scope="module")
def nf4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


def _gain(seed, K):
    # bf16 gains around 1 with a spread, as trained RMS weights are
    return synth.f32_bits_to_bf16((1.0 + 0.25 * synth.normal_f32(seed, 5, K)).astype(np.float32))


def _case(nf4, rows, K, eps, out, seed, scale=1.0):
    x = (synth.normal_f32(seed, 4, rows * K).reshape(rows, K) * np.float32(scale)).astype(np.float32)
    w = _gain(seed, K)
    y_ref, _ = oracle.rmsnorm(x, w, eps)
    xt = torch.from_numpy(x).cuda()
    wt = H.bf16_tensor(w)
    dtype = torch.float32 if out == "f32" else torch.bfloat16
    y = nf4.nf4_rmsnorm(xt, wt, eps, dtype=dtype)
    if out == "f32":
        got = y.cpu().numpy().astype(np.float64)
        extra = 0.0
    else:
        got = synth.bf16_to_f32(H.bf16_bits_of(y).reshape(-1)).reshape(rows, K).astype(np.float64)
        extra = H.ulp_bf16(y_ref.reshape(-1)).reshape(rows, K)
    bound = REL * np.abs(y_ref) + extra
    bad = np.argwhere(~(np.abs(got - y_ref) <= bound))
    assert bad.size == 0, f"{rows}x{K} eps={eps} {out}: {len(bad)} outside, first {bad[:3]}"
    return xt, wt, y


@pytest.mark.parametrize("rows,K", [(1, 2048), (1, 5120), (1, 11008), (7, 2048), (32, 5120), (1, 65536),
                                    (3, 1), (2, 33), (5, 64)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_rmsnorm_shapes(nf4, rows, K, out):
    _case(nf4, rows, K, 1e-6, out, 800 + rows + K)


@pytest.mark.parametrize("eps", [0.0, 0.5, 4.0])
def test_rmsnorm_eps(nf4, eps):
    # a large eps changes every value by a large factor: a dropped or misplaced
    # eps fails the bound
    _case(nf4, 4, 2048, eps, "f32", 810)


@pytest.mark.parametrize("scale", [2.0 ** -60, 2.0 ** 40])
def test_rmsnorm_extreme_magnitudes(nf4, scale):
    _case(nf4, 2, 2048, 0.0, "f32", 811, scale=scale)


def test_rmsnorm_in_place_and_deterministic(nf4):
    xt, wt, y = _case(nf4, 3, 5120, 1e-6, "f32", 820)
    x2 = xt.clone()
    nf4.nf4_rmsnorm(x2, wt, 1e-6, out=x2)  # in place over x
    assert torch.equal(x2, y)
    # identical rows give identical outputs, wherever they sit
    xs = xt[0:1].repeat(4, 1).contiguous()
    ys = nf4.nf4_rmsnorm(xs, wt, 1e-6, dtype=torch.float32)
    assert all(torch.equal(ys[i], y[0]) for i in range(4))


def test_rmsnorm_zero_row_is_zero(nf4):
    x = torch.zeros((2, 2048), device="cuda")
    w = H.bf16_tensor(_gain(830, 2048))
    y = nf4.nf4_rmsnorm(x, w, 1e-6, dtype=torch.float32)
    assert torch.count_nonzero(y).item() == 0


def test_rmsnorm_feeds_a_projection(nf4):
    # the decode step's order: RMS (bf16 out) -> projection with that bf16 x
    K, M = 2048, 2048
    x = synth.normal_f32(840, 4, K)
    w = _gain(840, K)
    xb = nf4.nf4_rmsnorm(torch.from_numpy(x).cuda(), H.bf16_tensor(w), 1e-6)
    xb_bits = H.bf16_bits_of(xb)
    y_ref_rms, _ = oracle.rmsnorm(x, w, 1e-6)
    want_bits = np.array([oracle.round_bf16(v) for v in y_ref_rms], np.uint16)
    # bf16 output: the oracle's own rounding or a neighbour (within one ulp)
    assert np.all(np.abs(xb_bits.astype(np.int32) - want_bits.astype(np.int32)) <= 1)
    codes, scales = H.quantized(841, 0, M, K)
    y_ref, S = oracle.gemv(codes, scales, xb_bits)
    y = nf4.nf4_gemv(H.weight_tensors(codes, scales), xb).cpu().numpy()
    H.assert_within(y, y_ref, S, what="projection of the normalized x")


def test_rmsnorm_errors(nf4):
    x = torch.ones(64, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nf4.NF4Error) as e:
        nf4.nf4_rmsnorm(x, w, -1.0)
    assert e.value.status == -1
    assert nf4.lib.nf4_rmsnorm(None, None, 1, 64, 0.0, None, 0, None) == -3  # NULL pointers
    with pytest.raises(nf4.NF4Error) as e:  # bf16 output over the fp32 input
        nf4.nf4_rmsnorm(x, w, 0.0, out=x.view(torch.bfloat16)[:64])
    assert e.value.status == -1
