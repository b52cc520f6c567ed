"""GPU parity of nf4_dequant_rows (NF4 embedding rows gathered and dequantized)
against the oracle: bit-exact, fp32 (one fp32 product per weight, as the
oracle) and bf16 (that product rounded to nearest even).  Out-of-range ids
write zero rows and are reported by nf4_check_device_errors as NF4_ERANGE; the
kernel checks every id, so no id can make it read outside the table.
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

    mod.nf4_check_device_errors()  # start from a clear error word
    return mod


def _run(nf4, E, ids, dtype):
    idt = torch.from_numpy(np.ascontiguousarray(ids, np.int64)).cuda()
    out = nf4.nf4_dequant_rows(E, idt, dtype=dtype)
    return out


@pytest.mark.parametrize("V,K,n", [(1, 64, 1), (1000, 512, 37), (300, 2048, 64), (20000, 2048, 33),
                                   (50, 11008, 5)])
def test_rows_bitexact(nf4, V, K, n):
    codes, scales = H.quantized(800 + V, 0, V, K)
    E = H.weight_tensors(codes, scales)
    ids = synth.token_ids(800 + V, 1, n, V)
    ids[n // 2] = ids[0]  # a repeated id
    f32, b16, bad = oracle.dequant_rows(codes, scales, ids)
    assert bad == 0
    got32 = _run(nf4, E, ids, torch.float32).cpu().numpy()
    assert np.array_equal(got32.view(np.uint32), f32.view(np.uint32))
    got16 = H.bf16_bits_of(_run(nf4, E, ids, torch.bfloat16))
    assert np.array_equal(got16.reshape(b16.shape), b16)
    nf4.nf4_check_device_errors()


def test_out_of_range_ids_give_zero_rows_and_erange(nf4):
    V, K = 100, 256
    codes, scales = H.quantized(810, 0, V, K)
    E = H.weight_tensors(codes, scales)
    ids = np.array([3, -1, 100, 99, 1 << 40, 0], np.int64)
    f32, _, bad = oracle.dequant_rows(codes, scales, ids)
    assert bad == 3
    got = _run(nf4, E, ids, torch.float32).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), f32.view(np.uint32))
    with pytest.raises(nf4.NF4Error, match="NF4_ERANGE"):
        nf4.nf4_check_device_errors()
    nf4.nf4_check_device_errors()  # read and cleared


def test_empty_and_argument_errors(nf4):
    codes, scales = H.quantized(820, 0, 10, 128)
    E = H.weight_tensors(codes, scales)
    out = nf4.nf4_dequant_rows(E, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert out.shape == (0, 128)
    ids = torch.zeros(4, dtype=torch.int64, device="cuda")
    buf = torch.empty(4 * 128 + 8, dtype=torch.float32, device="cuda")
    with pytest.raises(nf4.NF4Error, match="16-byte aligned"):
        nf4.nf4_dequant_rows(E, ids, out=buf[1:1 + 4 * 128].view(4, 128))
    with pytest.raises(TypeError):
        nf4.nf4_dequant_rows(E, ids, dtype=torch.float16)
