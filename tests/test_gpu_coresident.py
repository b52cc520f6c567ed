"""GPU parity of the bulk-copy GEMV sized for two blocks per SM
(NF4_TMA_CORESIDENT=1): one row group per block, at most half the SM's shared
memory, one block per SM, and the first stages copied before the dependency
wait so that a call's weight reads overlap the previous call's arithmetic.
Same bound against the oracle as every N=1 test, including calls launched
back to back on one stream (the overlap the mode exists for)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nf4_weight_quantized_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture
def nf4(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("NF4_TMA_CORESIDENT", "1")
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


@pytest.mark.parametrize("M,K", [(2048, 11008), (600, 5120), (300, 2048), (77, 1024), (5, 32768)])
@pytest.mark.parametrize("xd", ["f32", "bf16"])
def test_coresident_gemv(nf4, M, K, xd):
    seed = 700 + M
    codes, scales = H.quantized(seed, 0, M, K)
    x = H.make_x(seed, K, xd)
    y_ref, S = oracle.gemv(codes, scales, x)
    y = nf4.nf4_gemv(H.weight_tensors(codes, scales), H.x_tensor(x)).cpu().numpy()
    H.assert_within(y, y_ref, S, what=f"co-resident {M}x{K} {xd}")
    nf4.nf4_check_device_errors()


def test_coresident_down_is_paired_and_back_to_back(nf4):
    # the 3B down projection: the configuration must be the paired one, and
    # six calls on rotating weights launched back to back must all be right
    M, K = 2048, 11008
    assert "two blocks per SM" in nf4.nf4_describe_config(M, K)
    x = H.make_x(710, K, "bf16")
    xt = H.x_tensor(x)
    Ws, refs, outs = [], [], []
    for i in range(3):
        codes, scales = H.quantized(710 + i, 0, M, K)
        Ws.append(H.weight_tensors(codes, scales))
        r = synth.normal_f32(710 + i, 3, M)
        y64, _ = oracle.gemv_residual(codes, scales, x, r)
        _, S = oracle.gemv(codes, scales, x)
        refs.append((torch.from_numpy(r).cuda(), y64, S))
    torch.cuda.synchronize()
    for i in range(6):
        r, _, _ = refs[i % 3]
        outs.append(nf4.nf4_gemv_residual(Ws[i % 3], xt, r))
    torch.cuda.synchronize()
    for i in range(6):
        _, y64, S = refs[i % 3]
        y = outs[i].cpu().numpy()
        H.assert_within(y, y64, S, extra=H.ulp_f32(y64), what=f"back-to-back call {i}")
    nf4.nf4_check_device_errors()


@pytest.mark.parametrize("M,K", [(45, 2048), (700, 2048)])
def test_coresident_swiglu(nf4, M, K):
    seed = 720 + M
    gc, gs = H.quantized(seed, 0, M, K)
    uc, us = H.quantized(seed, 1, M, K)
    x = H.make_x(seed, K, "bf16")
    o64, _, g, u = oracle.gemv_swiglu(gc, gs, uc, us, x)
    _, Sg = oracle.gemv(gc, gs, x)
    _, Su = oracle.gemv(uc, us, x)
    out = nf4.nf4_gemv_swiglu(H.weight_tensors(gc, gs), H.weight_tensors(uc, us), H.x_tensor(x))
    of = synth.bf16_to_f32(H.bf16_bits_of(out)).astype(np.float64)
    assert np.all(np.abs(of - o64) <= H.swiglu_bound(g, u, Sg, Su) + H.ulp_bf16(o64))


def test_coresident_keeps_several_groups_for_short_rows(nf4):
    # K = 2048: a row group is one warp, so a paired block still holds several
    import re

    desc = nf4.nf4_describe_config(11008, 2048)
    assert "two blocks per SM" in desc, desc
    groups = int(re.search(r"(\d+) group\(s\)", desc).group(1))
    assert groups >= 2, desc
