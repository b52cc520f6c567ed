"""Pins for the CPU oracle: each check ties it to something other than itself.

Codebook: the closed form of the QLoRA NormalFloat construction evaluated with
scipy's inverse normal CDF (a library routine) and the table's invariants.
Encoder: exact rational brute force, round trip, error bound, zero block.
GEMV: hand-computed worked examples (tests/golden/worked_examples.txt), each
code reading its own level (one-hot x against scipy's closed form), exact
sums via math.fsum, numpy float64 matmul, power-of-two linearity, the zero level.
Epilogues: residual / SwiGLU / argmax reduce to the GEMV plus their definitions;
fused q/k/v: a worked example with distinct closed-form values per segment, zero
scales giving exactly the bias, row sampling across the segment boundaries;
embedding rows: a worked example with exact values and bf16 bits, out-of-range
ids giving zero rows, bf16 equal to round-to-nearest-even on the bit pattern;
argmax ties go to the lowest index ("golang.design/x/accel/tensor", func Argmax);
SwiGLU with gate/up rows interleaved: a worked example using silu(0) = 0 and
silu(z) - silu(-z) = z, and equality with the two-matrix SwiGLU.
Chunk: equals the GEMV exactly when every W_hat is representable in bf16, and
otherwise stays within the bf16 rounding bound of the weights.
RMSNorm: closed forms (a row whose mean square is a perfect square, an eps that
completes one, rows normalized separately), the bf16 gain bits, power-of-two
scale invariance and unit root mean square of the output.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from nf4_weight_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


# ------------------------------------------------------------------ codebook

def test_codebook_invariants(cb):
    assert cb.dtype == np.float32 and cb.shape == (16,)
    assert np.all(np.diff(cb.astype(np.float64)) > 0)
    assert cb[0] == -1.0 and cb[7] == 0.0 and cb[15] == 1.0
    assert np.sum(cb > 0) == 8 and np.sum(cb < 0) == 7  # asymmetric: 8 positive, 7 negative


def test_codebook_closed_form_matches_scipy(cb):
    ndtri = pytest.importorskip("scipy.special").ndtri
    d = 0.5 * (1 / 32 + 1 / 30)
    pos = ndtri(1 - d - np.arange(8) * (0.5 - d) / 8)
    neg = ndtri(d + np.arange(7) * (0.5 - d) / 7)
    ref = (np.sort(np.concatenate([pos, neg, [0.0]])) / ndtri(1 - d)).astype(np.float32)
    assert np.array_equal(ref.view(np.uint32), cb.view(np.uint32))


def test_codebook_values_to_1e6(cb):
    # the 16 levels, 7 decimals (float64 evaluation of the construction)
    printed = [-1.0, -0.6961928, -0.5250729, -0.3949175, -0.2844413, -0.1847734, -0.0910500, 0.0,
               0.0795803, 0.1609302, 0.2461123, 0.3379152, 0.4407097, 0.5626170, 0.7229568, 1.0]
    assert np.max(np.abs(cb.astype(np.float64) - np.array(printed))) < 1e-6


# ------------------------------------------------------------------- encoder

def _exact_nearest(cb, w, s):
    """Nearest level to w/s in exact rationals, ties to the lower index."""
    if s == 0:
        return 7
    v = Fraction(float(w)) / Fraction(float(s))
    best, best_d = None, None
    for i, c in enumerate(cb):
        dd = abs(v - Fraction(float(c)))
        if best is None or dd < best_d:
            best, best_d = i, dd
    return best


def _unpack(codes, K):
    lo = codes & 0x0F
    hi = codes >> 4
    out = np.empty((codes.shape[0], K), np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _pack(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_encoder_exact_bruteforce(oracle_mod, cb):
    g = np.random.Generator(np.random.PCG64(11))
    W = (g.standard_normal((3, 128)) * 0.02).astype(np.float32)
    # plant exact ties: values at the midpoint of two levels times the block absmax
    s = np.float32(np.max(np.abs(W[0, :64])))
    for i in range(15):
        mid = (Fraction(float(cb[i])) + Fraction(float(cb[i + 1]))) / 2 * Fraction(float(s))
        f = np.float32(float(mid))
        if Fraction(float(f)) == mid and abs(f) < s:
            W[0, 2 + i] = f
    codes, scales = oracle_mod.quantize(W)
    cu = _unpack(codes, 128)
    for m in range(3):
        for b in range(2):
            blk = W[m, 64 * b:64 * b + 64]
            s = np.float32(np.max(np.abs(blk)))
            assert scales[m, b] == s
            for j in range(64):
                assert cu[m, 64 * b + j] == _exact_nearest(cb, blk[j], s), (m, b, j)


def test_encoder_ties_go_low(oracle_mod, cb):
    # a block whose absmax is 1 and which holds every exact midpoint of the table
    # that fp32 can represent: each must map to the lower of its two levels
    W = np.zeros((1, 64), np.float32)
    W[0, 0] = 1.0
    planted = []
    for i in range(15):
        mid = (Fraction(float(cb[i])) + Fraction(float(cb[i + 1]))) / 2
        f = np.float32(float(mid))
        if Fraction(float(f)) == mid:
            W[0, 1 + i] = f
            planted.append((1 + i, i))
    assert planted, "no representable midpoint"
    codes, _ = oracle_mod.quantize(W)
    cu = _unpack(codes, 64)
    for k, lower in planted:
        assert cu[0, k] == lower


def test_midpoint_products_are_exact(cb):
    # the encoder compares w against mid_i * s in float64; check that both the
    # midpoints and their products with fp32 scales carry at most 53 bits
    g = np.random.Generator(np.random.PCG64(5))
    scales = np.abs(g.standard_normal(200)).astype(np.float32)
    for i in range(15):
        mid = (Fraction(float(cb[i])) + Fraction(float(cb[i + 1]))) / 2
        assert Fraction((float(cb[i]) + float(cb[i + 1])) / 2) == mid
        for s in scales:
            assert Fraction(float(mid) * float(s)) == mid * Fraction(float(s))


def test_zero_block(oracle_mod):
    W = np.zeros((2, 128), np.float32)
    W[0, 64:] = -0.0
    W[1, :64] = np.linspace(-1, 1, 64, dtype=np.float32)
    codes, scales = oracle_mod.quantize(W)
    assert np.all(codes[0] == 0x77) and np.all(scales[0] == 0.0)
    assert np.all(codes[1, 32:] == 0x77) and scales[1, 1] == 0.0
    assert scales[1, 0] == 1.0


def test_roundtrip(oracle_mod, cb):
    g = np.random.Generator(np.random.PCG64(3))
    M, K = 8, 256
    c = g.integers(0, 16, size=(M, K)).astype(np.uint8)
    c[:, ::64] = g.choice([0, 15], size=(M, K // 64))  # every block holds a +-1 level
    s = (np.abs(g.standard_normal((M, K // 64))) * 0.05 + 1e-3).astype(np.float32)
    codes = _pack(c)
    W_hat = oracle_mod.dequant(codes, s)
    codes2, s2 = oracle_mod.quantize(W_hat)
    assert np.array_equal(codes2, codes)
    assert np.array_equal(s2, s)


def test_dequant_definition(oracle_mod, cb):
    g = np.random.Generator(np.random.PCG64(4))
    M, K = 4, 128
    c = g.integers(0, 16, size=(M, K)).astype(np.uint8)
    s = g.standard_normal((M, K // 64)).astype(np.float32)
    W_hat = oracle_mod.dequant(_pack(c), s)
    ref = (cb[c] * np.repeat(s, 64, axis=1)).astype(np.float32)  # fp32 product
    assert np.array_equal(W_hat.view(np.uint32), ref.view(np.uint32))


def test_quantization_error_bound(oracle_mod, cb):
    W = synth.weights(7, 0, 16, 512)
    codes, scales = oracle_mod.quantize(W)
    W_hat = oracle_mod.dequant(codes, scales).astype(np.float64)
    half_gap = np.max(np.diff(cb.astype(np.float64))) / 2  # 0.1519...
    assert abs(half_gap - 0.15190) < 1e-4
    s = np.repeat(scales.astype(np.float64), 64, axis=1)
    assert np.all(np.abs(W.astype(np.float64) - W_hat) <= half_gap * s * (1 + 1e-6))


# ---------------------------------------------------------------------- GEMV

def _parse_golden():
    cases = []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, _, rest = line.partition(" ")
            if head == "case":
                name, kk = rest.split()
                cur = {"name": name, "K": int(kk.split("=")[1]), "rows": [], "x": None, "y": None}
                cases.append(cur)
            elif head == "row":
                blocks, scales = rest.split("|")
                cur["rows"].append((blocks.split(), [float(v) for v in scales.split()]))
            elif head == "x":
                cur["x"] = rest
            elif head == "y":
                cur["y"] = [float(v) for v in rest.split()]
    return cases


def _build_case(case):
    K = case["K"]
    M = len(case["rows"])
    c = np.zeros((M, K), np.uint8)
    s = np.zeros((M, K // 64), np.float32)
    for m, (blocks, scales) in enumerate(case["rows"]):
        for b, tok in enumerate(blocks):
            if tok.startswith("alt"):
                a, bb = (int(v) for v in tok[3:].split(","))
                c[m, 64 * b:64 * b + 64:2] = a
                c[m, 64 * b + 1:64 * b + 64:2] = bb
            else:
                c[m, 64 * b:64 * b + 64] = int(tok[1:])
        s[m] = scales
    rule = case["x"].split()
    k = np.arange(K)
    if rule[0] == "ones":
        x = np.ones(K)
    elif rule[0] == "k":
        x = k.astype(np.float64)
    elif rule[0] == "steps":
        vals = [float(v) for v in rule[1].split(",")]
        x = np.array([vals[i // 64] for i in k])
    elif rule[0] == "onehot":
        x = np.zeros(K)
        x[int(rule[1])] = 1.0
    else:
        raise ValueError(rule)
    return _pack(c), s, x.astype(np.float32)


@pytest.mark.parametrize("case", _parse_golden(), ids=lambda c: c["name"])
def test_worked_examples(oracle_mod, case):
    codes, scales, x = _build_case(case)
    y, _ = oracle_mod.gemv(codes, scales, x)
    assert list(y) == case["y"]
    # same activation as bf16 (all values here are exact in bf16)
    xb = synth.f32_bits_to_bf16(x)
    assert np.array_equal(synth.bf16_to_f32(xb), x)
    yb, _ = oracle_mod.gemv(codes, scales, xb)
    assert list(yb) == case["y"]


def test_sum_of_levels(oracle_mod, cb):
    # codes 0..15 repeated four times, scale 1, x = 1: y = 4 * sum(cb)
    c = np.tile(np.arange(16, dtype=np.uint8), 4)[None, :]
    y, S = oracle_mod.gemv(_pack(c), np.ones((1, 1), np.float32), np.ones(64, np.float32))
    assert y[0] == math.fsum(4 * [float(v) for v in cb])
    assert S[0] == math.fsum(4 * [abs(float(v)) for v in cb])


def test_each_code_reads_its_own_level(oracle_mod):
    # A permuted table would keep the sum of levels; this pins code -> level.
    # Row c holds code c everywhere (both nibbles), scale 2^-3 in block 0 and
    # 3 in block 1.  x = e_j picks one weight: y_c = level_c * scale, with the
    # levels from the closed form of the construction (scipy's inverse normal
    # CDF, independent of the oracle's bisection), rounded to fp32, times a
    # scale; the fp32 product is exact for 2^-3 and rounded once for 3.
    ndtri = pytest.importorskip("scipy.special").ndtri
    d = 0.5 * (1 / 32 + 1 / 30)
    lv = np.sort(np.concatenate([ndtri(1 - d - np.arange(8) * (0.5 - d) / 8),
                                 ndtri(d + np.arange(7) * (0.5 - d) / 7), [0.0]])) / ndtri(1 - d)
    lv = lv.astype(np.float32)
    K = 128
    codes = np.repeat((np.arange(16, dtype=np.uint8) * 0x11)[:, None], K // 2, axis=1)
    scales = np.tile(np.array([[0.125, 3.0]], np.float32), (16, 1))
    for j, s in ((0, 0.125), (1, 0.125), (63, 0.125), (64, 3.0), (127, 3.0)):
        x = np.zeros(K, np.float32)
        x[j] = 1.0
        y, _ = oracle_mod.gemv(codes, scales, x)
        want = (lv * np.float32(s)).astype(np.float64)  # one fp32 rounding of the product
        assert np.array_equal(y, want), (j, y, want)


def test_gemv_exact_sum(oracle_mod):
    W = synth.weights(9, 0, 6, 1024)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_bf16(9, 1, 1024)
    y, S = oracle_mod.gemv(codes, scales, x)
    W_hat = oracle_mod.dequant(codes, scales).astype(np.float64)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    for m in range(6):
        terms = W_hat[m] * xf  # exact: fp32 x bf16 products fit in float64
        assert abs(y[m] - math.fsum(terms)) <= 1e-13 * S[m]
        assert abs(S[m] - math.fsum(np.abs(terms))) <= 1e-13 * S[m]


def test_gemv_vs_numpy_matmul(oracle_mod):
    W = synth.weights(10, 0, 256, 512)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_f32(10, 1, 512)
    y, S = oracle_mod.gemv(codes, scales, x)
    ref = oracle_mod.dequant(codes, scales).astype(np.float64) @ x.astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-12 * S)


def test_gemv_row_subset(oracle_mod):
    W = synth.weights(12, 0, 64, 256)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_f32(12, 1, 256)
    y_all, S_all = oracle_mod.gemv(codes, scales, x)
    rows = np.array([63, 0, 17, 17, 5])
    y, S = oracle_mod.gemv(codes, scales, x, rows=rows)
    assert np.array_equal(y, y_all[rows]) and np.array_equal(S, S_all[rows])


def test_gemv_linearity_power_of_two(oracle_mod):
    W = synth.weights(13, 0, 32, 256)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_f32(13, 1, 256)
    y, _ = oracle_mod.gemv(codes, scales, x)
    for a in (2.0, 0.25, -8.0):
        ya, _ = oracle_mod.gemv(codes, scales, (x * a).astype(np.float32))
        assert np.array_equal(ya, y * a)


def test_zero_level_rows(oracle_mod):
    g = np.random.Generator(np.random.PCG64(14))
    M, K = 4, 192
    codes = np.full((M, K // 2), 0x77, np.uint8)
    scales = (g.standard_normal((M, K // 64)) * 100).astype(np.float32)
    x = g.standard_normal(K).astype(np.float32)
    y, S = oracle_mod.gemv(codes, scales, x)
    assert np.all(y == 0.0) and np.all(S == 0.0)
    r = g.standard_normal(M).astype(np.float32)
    y64, y32 = oracle_mod.gemv_residual(codes, scales, x, r)
    assert np.array_equal(y32, r)


# ----------------------------------------------------------------- epilogues

def test_residual(oracle_mod):
    W = synth.weights(15, 0, 64, 256)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_bf16(15, 1, 256)
    r = synth.normal_f32(15, 2, 64)
    y, _ = oracle_mod.gemv(codes, scales, x)
    y64, y32 = oracle_mod.gemv_residual(codes, scales, x, r)
    assert np.array_equal(y64, y + r.astype(np.float64))
    assert np.array_equal(y32, (y + r.astype(np.float64)).astype(np.float32))


def _exact_bf16_round(v: float) -> int:
    """bf16 bits of a finite nonzero double by exact rational rounding (ties to even)."""
    if v == 0:
        return 0x8000 if math.copysign(1, v) < 0 else 0
    sign = 0x8000 if v < 0 else 0
    a = Fraction(abs(v))
    e = math.floor(math.log2(abs(v)))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 7, -133)
    scaled = a / Fraction(2) ** q
    r = math.floor(scaled)
    rem = scaled - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    val = float(Fraction(r) * Fraction(2) ** q)
    return sign | int(np.array([val], np.float32).view(np.uint32)[0] >> 16)


def test_round_bf16(oracle_mod):
    g = np.random.Generator(np.random.PCG64(16))
    vals = list(g.standard_normal(300) * 10.0 ** g.integers(-30, 30, 300))
    # exact ties between two bf16 neighbours (odd and even last bits) and extremes
    vals += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.5e-40, 2.0 ** -133 * 1.5]
    for v in vals:
        assert oracle_mod.round_bf16(v) == _exact_bf16_round(v), v
    assert oracle_mod.round_bf16(3.4e38) == 0x7F80  # rounds past the largest bf16


def test_swiglu(oracle_mod):
    M, K = 48, 256
    Wg = synth.weights(17, 0, M, K)
    Wu = synth.weights(17, 1, M, K)
    Wg[3] = 0.0  # a zero gate row: silu(0) = 0
    gc, gs = oracle_mod.quantize(Wg)
    uc, us = oracle_mod.quantize(Wu)
    x = synth.normal_bf16(17, 2, K)
    out64, outbf, g, u = oracle_mod.gemv_swiglu(gc, gs, uc, us, x)
    yg, _ = oracle_mod.gemv(gc, gs, x)
    yu, _ = oracle_mod.gemv(uc, us, x)
    assert np.array_equal(g, yg) and np.array_equal(u, yu)
    assert out64[3] == 0.0 and outbf[3] in (0, 0x8000)
    # silu(z) = z * sigmoid(z): compare with an independent logistic form
    ref = g * (0.5 * (1.0 + np.tanh(0.5 * g))) * u
    assert np.all(np.abs(out64 - ref) <= 1e-13 * (np.abs(ref) + 1e-30))
    for i in range(M):
        assert outbf[i] == _exact_bf16_round(out64[i]) or out64[i] == 0.0


def test_swiglu_limits(oracle_mod):
    # large positive gate: silu(g) -> g; large negative gate: silu(g) -> 0
    K = 64
    gc = np.full((2, 32), 0xFF, np.uint8)  # all +1
    gs = np.array([[1.0], [-1.0]], np.float32)  # row 0: +64, row 1: -64 (x = 1)
    uc = np.full((2, 32), 0xFF, np.uint8)
    us = np.array([[0.5], [0.5]], np.float32)  # u = 32
    x = np.ones(K, np.float32)
    out64, _, g, u = oracle_mod.gemv_swiglu(gc, gs, uc, us, x)
    assert g[0] == 64 and g[1] == -64 and u[0] == 32
    assert abs(out64[0] - 64 * 32) < 1e-9
    assert abs(out64[1]) < 1e-20


def test_argmax_bruteforce_and_ties(oracle_mod):
    M, K = 300, 256
    W = synth.weights(18, 0, M, K)
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_bf16(18, 1, K)
    l64, l32, idx = oracle_mod.gemv_argmax(codes, scales, x)
    y, _ = oracle_mod.gemv(codes, scales, x)
    assert np.array_equal(l64, y)
    assert np.array_equal(l32, y.astype(np.float32))
    assert idx == int(np.argmax(y)) and y[idx] == y.max()
    # duplicate the winning row before and after it: the lowest copy wins
    best = idx
    lo, hi = best // 2, min(M - 1, best + 7)
    codes2, scales2 = codes.copy(), scales.copy()
    for r in (lo, hi):
        codes2[r], scales2[r] = codes[best], scales[best]
    _, _, idx2 = oracle_mod.gemv_argmax(codes2, scales2, x)
    assert idx2 == min(lo, best)


def test_argmax_all_equal():
    import oracle

    codes = np.full((10, 32), 0x77, np.uint8)
    scales = np.ones((10, 1), np.float32)
    _, _, idx = oracle.gemv_argmax(codes, scales, np.ones(64, np.float32))
    assert idx == 0


# --------------------------------------------------------------------- chunk

def test_chunk_equals_gemv_when_weights_are_bf16_exact(oracle_mod):
    g = np.random.Generator(np.random.PCG64(19))
    M, K, N = 24, 256, 5
    c = g.choice([0, 7, 15], size=(M, K)).astype(np.uint8)  # levels -1, 0, +1
    s = (2.0 ** g.integers(-8, 3, size=(M, K // 64))).astype(np.float32)
    codes = _pack(c)
    X = synth.normal_bf16(19, 1, N * K).reshape(N, K)
    Y, S = oracle_mod.gemm_chunk(codes, s, X)
    for n in range(N):
        y, Sg = oracle_mod.gemv(codes, s, X[n])
        assert np.array_equal(Y[n], y) and np.array_equal(S[n], Sg)


def test_chunk_bf16_weight_bound(oracle_mod):
    W = synth.weights(20, 0, 40, 512)
    codes, scales = oracle_mod.quantize(W)
    X = synth.normal_bf16(20, 1, 3 * 512).reshape(3, 512)
    Y, S = oracle_mod.gemm_chunk(codes, scales, X)
    for n in range(3):
        y, Sg = oracle_mod.gemv(codes, scales, X[n])
        # each weight moves by at most 2^-9 relative when rounded to bf16
        assert np.all(np.abs(Y[n] - y) <= 2.0 ** -9 * Sg * (1 + 1e-9))
        assert np.any(Y[n] != y)  # the rounding is really applied
    rows = np.array([39, 2])
    Yr, _ = oracle_mod.gemm_chunk(codes, scales, X, rows=rows)
    assert np.array_equal(Yr, Y[:, rows])


def test_chunk_explicit_bf16_products(oracle_mod, cb):
    # small case spelled out: bf16(W_hat) via numpy rounding of the fp32 W_hat
    W = synth.weights(21, 0, 3, 64)
    codes, scales = oracle_mod.quantize(W)
    W_hat = oracle_mod.dequant(codes, scales)
    Wb = synth.bf16_to_f32(synth.f32_bits_to_bf16(W_hat)).astype(np.float64)
    X = synth.normal_bf16(21, 1, 2 * 64).reshape(2, 64)
    Y, _ = oracle_mod.gemm_chunk(codes, scales, X)
    Xf = synth.bf16_to_f32(X).astype(np.float64)
    for n in range(2):
        for m in range(3):
            assert abs(Y[n, m] - math.fsum(Wb[m] * Xf[n])) <= 1e-14 * np.sum(np.abs(Wb[m] * Xf[n]))


# ------------------------------------------------------------- fused q/k/v


def _const_codes(M, K, byte):
    return np.full((M, K // 2), byte, np.uint8)


def test_qkv_worked_example(oracle_mod, cb):
    # q rows: every code 15 (level +1); k rows: code 0 (level -1); v rows: code 7
    # (level 0).  Scale 0.5 everywhere, x = 1 (K = 128), bias b = row index / 4.
    # Then y_q = 128 * 0.5 + b = 64 + b, y_k = -64 + b, y_v = b, exactly.
    assert cb[15] == 1.0 and cb[0] == -1.0 and cb[7] == 0.0
    K = 128
    Mq, Mk, Mv = 6, 2, 3
    parts = []
    for M, byte in ((Mq, 0xFF), (Mk, 0x00), (Mv, 0x77)):
        bias = (np.arange(M, dtype=np.float32) / 4).astype(np.float32)
        parts.append((_const_codes(M, K, byte), np.full((M, K // 64), 0.5, np.float32), bias))
    y, S = oracle_mod.gemv_qkv(parts, np.ones(K, np.float32))
    want = [64 + i / 4 for i in range(Mq)] + [-64 + i / 4 for i in range(Mk)] + [i / 4 for i in range(Mv)]
    assert list(y) == want
    assert list(S) == [64 + i / 4 for i in range(Mq)] + [64 + i / 4 for i in range(Mk)] + [i / 4 for i in range(Mv)]
    # no bias on k: k rows become exactly -64
    parts[1] = (parts[1][0], parts[1][1], None)
    y2, _ = oracle_mod.gemv_qkv(parts, np.ones(K, np.float32))
    assert list(y2[Mq:Mq + Mk]) == [-64.0, -64.0]
    assert np.array_equal(y2[:Mq], y[:Mq]) and np.array_equal(y2[Mq + Mk:], y[Mq + Mk:])


def test_qkv_zero_scales_give_the_bias(oracle_mod):
    K = 256
    parts = []
    for t, M in enumerate((5, 3, 4)):
        codes, _ = oracle_mod.quantize(synth.weights(70 + t, 0, M, K))
        bias = synth.normal_f32(70 + t, 1, M)
        parts.append((codes, np.zeros((M, K // 64), np.float32), bias))
    y, S = oracle_mod.gemv_qkv(parts, synth.normal_bf16(70, 2, K))
    b = np.concatenate([p[2] for p in parts]).astype(np.float64)
    assert np.array_equal(y, b) and np.array_equal(S, np.abs(b))


def test_qkv_rows_span_segments(oracle_mod):
    # sampled rows across the q/k and k/v boundaries equal the unsampled ones,
    # and each segment equals the exact sum of its own dequantized products
    K = 512
    parts = []
    for t, M in enumerate((7, 2, 5)):
        codes, scales = oracle_mod.quantize(synth.weights(80 + t, 0, M, K))
        parts.append((codes, scales, synth.normal_f32(80 + t, 1, M)))
    x = synth.normal_bf16(80, 2, K)
    y, S = oracle_mod.gemv_qkv(parts, x)
    rows = [13, 0, 6, 7, 8, 9]
    ys, Ss = oracle_mod.gemv_qkv(parts, x, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(Ss, S[rows])
    xf = synth.bf16_to_f32(x).astype(np.float64)
    base = 0
    for codes, scales, bias in parts:
        W_hat = oracle_mod.dequant(codes, scales).astype(np.float64)
        for m in range(codes.shape[0]):
            terms = W_hat[m] * xf
            assert abs(y[base + m] - (math.fsum(terms) + float(bias[m]))) <= 1e-13 * S[base + m]
        base += codes.shape[0]


# ------------------------------------------------------- NF4 embedding rows


def test_dequant_rows_worked_example(oracle_mod, cb):
    # row 0: bytes 0xF0 (low nibble 0 -> -1, high nibble 15 -> +1), scale 2.5;
    # row 1: bytes 0x77 (level 0); row 2: bytes 0x0F (+1, -1), scale -0.5
    K = 64
    codes = np.stack([np.full(K // 2, 0xF0, np.uint8), np.full(K // 2, 0x77, np.uint8),
                      np.full(K // 2, 0x0F, np.uint8)])
    scales = np.array([[2.5], [7.0], [-0.5]], np.float32)
    f32, b16, bad = oracle_mod.dequant_rows(codes, scales, np.array([2, 0, 1, 0]))
    assert bad == 0
    assert list(f32[1][:4]) == [-2.5, 2.5, -2.5, 2.5] and np.array_equal(f32[1], f32[3])
    assert list(f32[0][:4]) == [-0.5, 0.5, -0.5, 0.5]
    assert np.all(f32[2] == 0.0)
    assert list(b16[1][:2]) == [0xC020, 0x4020]  # -2.5, 2.5 in bf16
    assert list(b16[0][:2]) == [0xBF00, 0x3F00]  # -0.5, 0.5


def test_dequant_rows_out_of_range_ids_are_zero(oracle_mod):
    codes, scales = oracle_mod.quantize(synth.weights(90, 0, 5, 128))
    f32, b16, bad = oracle_mod.dequant_rows(codes, scales, np.array([-1, 5, 4, 1 << 40]))
    assert bad == 3
    assert np.all(f32[[0, 1, 3]] == 0) and np.all(b16[[0, 1, 3]] == 0)
    assert np.array_equal(f32[2], oracle_mod.dequant(codes, scales)[4])


def test_dequant_rows_bf16_is_round_to_nearest_even(oracle_mod):
    codes, scales = oracle_mod.quantize(synth.weights(91, 0, 64, 512))
    ids = synth.token_ids(91, 1, 40, 64)
    f32, b16, bad = oracle_mod.dequant_rows(codes, scales, ids)
    assert bad == 0
    full = oracle_mod.dequant(codes, scales)
    assert np.array_equal(f32, full[ids])
    # bf16 rounding written out on the bit pattern (finite values)
    u = f32.view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b16, rne)


# ------------------------------------------- SwiGLU, gate/up rows interleaved
# "gizai:tensor/lazy", method Lazy.gluIn: output column c is silu(v[2c]) times
# v[2c + 1], v the product of one matrix whose rows alternate gate and up.


def test_glu_interleaved_worked_example(oracle_mod, cb):
    # K = 64, x = 1.  Rows (level, scale): 0: (+1, 0.5) -> g0 = 32;
    # 1: (-1, 0.25) -> u0 = -16; 2: (0, 9) -> g1 = 0; 3: (+1, 2) -> u1 = 128;
    # 4: (-1, 0.5) -> g2 = -32; 5: (-1, 0.25) -> u2 = -16.
    # silu(0) = 0, so out1 = 0 exactly.  silu(z) - silu(-z) = z for every z
    # (z s(z) + z s(-z) = z, s the logistic function), so out0 - out2 = 32 u0
    # = -512 up to float64 rounding of the two products.  Applying silu to the
    # up rows instead, or pairing rows (2c+1, 2c+2), breaks both.
    assert cb[15] == 1.0 and cb[0] == -1.0 and cb[7] == 0.0
    K = 64
    byte = {1: 0xFF, -1: 0x00, 0: 0x77}
    spec = [(1, 0.5), (-1, 0.25), (0, 9.0), (1, 2.0), (-1, 0.5), (-1, 0.25)]
    codes = np.stack([np.full(K // 2, byte[lv], np.uint8) for lv, _ in spec])
    scales = np.array([[s] for _, s in spec], np.float32)
    out, obf, g, u = oracle_mod.gemv_glu_interleaved(codes, scales, np.ones(K, np.float32))
    assert list(g) == [32.0, 0.0, -32.0] and list(u) == [-16.0, 128.0, -16.0]
    assert out[1] == 0.0 and obf[1] in (0, 0x8000)
    assert abs((out[0] - out[2]) - (-512.0)) <= 1e-12
    # out0 = -16 * 32 / (1 + e^-32): within 1e-13 of -512; bf16 of it is -512
    assert abs(out[0] + 512.0) < 1e-10 and obf[0] == 0xC400
    assert 0.0 < out[2] < 1e-10  # -16 * silu(-32), silu(-32) ~ -4e-13


def test_glu_interleaved_equals_two_matrices(oracle_mod):
    # the interleaved layout is the two-matrix SwiGLU with gate = even rows and
    # up = odd rows, value for value
    M, K = 40, 320
    Wg = synth.weights(95, 0, M, K)
    Wu = synth.weights(95, 1, M, K)
    W = np.empty((2 * M, K), np.float32)
    W[0::2], W[1::2] = Wg, Wu
    codes, scales = oracle_mod.quantize(W)
    x = synth.normal_bf16(95, 2, K)
    out, obf, g, u = oracle_mod.gemv_glu_interleaved(codes, scales, x)
    ref = oracle_mod.gemv_swiglu(codes[0::2], scales[0::2], codes[1::2], scales[1::2], x)
    for a, b in zip((out, obf, g, u), ref):
        assert np.array_equal(a, b)
    cols = [M - 1, 0, 17, 17]
    sub = oracle_mod.gemv_glu_interleaved(codes, scales, x, cols=cols)
    for a, b in zip(sub, (out, obf, g, u)):
        assert np.array_equal(a, b[cols])


def test_glu_interleaved_rejects_bad_shapes(oracle_mod):
    K = 64
    codes = np.full((3, K // 2), 0x77, np.uint8)
    scales = np.ones((3, 1), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.gemv_glu_interleaved(codes, scales, np.ones(K, np.float32))  # odd row count
    with pytest.raises(ValueError):
        oracle_mod.gemv_glu_interleaved(codes[:2], scales[:2], np.ones(K, np.float32), cols=[1])


# ------------------------------------------------------------------ rmsnorm
# "Decode V2 -- resident executor", section 3: x * rsqrt(mean(x^2) + eps) * w,
# w bf16 [hidden]; "golang.design/x/accel/tensor", func RMSNorm: each row by
# its own root mean square.

BF16_ONE, BF16_TWO, BF16_MINUS_HALF, BF16_QUARTER = 0x3F80, 0x4000, 0xBF00, 0x3E80


def test_rmsnorm_worked_example(oracle_mod):
    # mean((1, 7, 1, 7)^2) = 100 / 4 = 25, so every value is divided by 5; a
    # sum instead of a mean (10), sqrt instead of rsqrt, or a dropped gain fails
    x = np.array([1.0, 7.0, 1.0, 7.0], np.float32)
    w = np.array([BF16_ONE, BF16_TWO, BF16_MINUS_HALF, BF16_QUARTER], np.uint16)
    y, ms = oracle_mod.rmsnorm(x, w, 0.0)
    assert ms == 25.0
    assert np.allclose(y, [0.2, 2.8, -0.1, 0.35], rtol=0, atol=1e-15)


def test_rmsnorm_eps_inside_the_root(oracle_mod):
    # mean square 1, eps 3: 1 / sqrt(1 + 3) = 1/2 exactly (eps dropped gives 1,
    # eps added outside the root gives 1 / 1 + 3 = 4)
    x = np.ones(8, np.float32)
    w = np.full(8, BF16_TWO, np.uint16)
    y, ms = oracle_mod.rmsnorm(x, w, 3.0)
    assert ms == 1.0 and np.all(y == 1.0)


def test_rmsnorm_rows_are_separate(oracle_mod):
    x = np.array([[2.0, -2.0, 2.0, 2.0], [1.0, 7.0, 1.0, 7.0]], np.float32)
    w = np.full(4, BF16_ONE, np.uint16)
    y, ms = oracle_mod.rmsnorm(x, w, 0.0)
    assert list(ms) == [4.0, 25.0]
    assert np.all(y[0] == [1.0, -1.0, 1.0, 1.0])
    assert np.allclose(y[1], [0.2, 1.4, 0.2, 1.4], rtol=0, atol=1e-15)


def test_rmsnorm_scale_invariance_and_unit_rms(oracle_mod):
    x = synth.normal_f32(77, 0, 3 * 2048).reshape(3, 2048)
    w = np.full(2048, BF16_ONE, np.uint16)
    y, _ = oracle_mod.rmsnorm(x, w, 0.0)
    # with eps = 0 and a unit gain every row has root mean square 1
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=0, atol=1e-12)
    # power-of-two scaling of x is exact in fp32 and cancels
    for e in (-20, -3, 5, 30):
        y2, _ = oracle_mod.rmsnorm(x * np.float32(2.0 ** e), w, 0.0)
        assert np.allclose(y2, y, rtol=1e-14, atol=0)


def test_rmsnorm_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.rmsnorm(np.ones(4, np.float32), np.ones(3, np.uint16), 0.0)
    with pytest.raises(ValueError):
        oracle_mod.rmsnorm(np.ones(4, np.float32), np.ones(4, np.uint16), -1.0)


def test_ref_entry_points_round_the_float64_results_once(oracle_mod):
    # nf4_ref_* take the library's arguments with host pointers; each result is
    # the float64 definition rounded once to the output type
    import ctypes

    oracle = oracle_mod
    lib = oracle.load()
    W_ = oracle.RefWeight
    M, K = 40, 256
    W = synth.weights(990, 0, M, K)
    codes, scales = oracle.quantize(W)
    c2 = np.zeros_like(codes)
    s2 = np.zeros_like(scales)
    assert lib.nf4_ref_quantize(W.ctypes.data, M, K, c2.ctypes.data, s2.ctypes.data) == 0
    assert np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint32), scales.view(np.uint32))
    w = W_.of(codes, scales)
    P = ctypes.byref
    for xt, x in ((0, synth.normal_f32(990, 1, K)), (1, synth.normal_bf16(990, 1, K))):
        y64, _ = oracle.gemv(codes, scales, x)
        y = np.zeros(M, np.float32)
        assert lib.nf4_ref_gemv(P(w), x.ctypes.data, xt, y.ctypes.data) == 0
        assert np.array_equal(y, y64.astype(np.float32))
        r = synth.normal_f32(990, 2, M)
        ry = r.copy()
        assert lib.nf4_ref_gemv_residual(P(w), x.ctypes.data, xt, ry.ctypes.data, ry.ctypes.data) == 0  # in place
        assert np.array_equal(ry, oracle.gemv_residual(codes, scales, x, r)[1])
        l64, l32, idx = oracle.gemv_argmax(codes, scales, x)
        lg = np.zeros(M, np.float32)
        ix = np.zeros(1, np.int64)
        assert lib.nf4_ref_gemv_argmax(P(w), x.ctypes.data, xt, lg.ctypes.data, ix.ctypes.data) == 0
        assert np.array_equal(lg, l32) and int(ix[0]) == idx
    x = synth.normal_bf16(991, 1, K)
    gc, gs = oracle.quantize(synth.weights(991, 1, M, K))
    out = np.zeros(M, np.uint16)
    assert lib.nf4_ref_gemv_swiglu(P(w), P(W_.of(gc, gs)), x.ctypes.data, 1, out.ctypes.data) == 0
    assert np.array_equal(out, oracle.gemv_swiglu(codes, scales, gc, gs, x)[1])
    out2 = np.zeros(M // 2, np.uint16)
    assert lib.nf4_ref_gemv_glu_interleaved(P(w), x.ctypes.data, 1, out2.ctypes.data) == 0
    assert np.array_equal(out2, oracle.gemv_glu_interleaved(codes, scales, x)[1])
    bq = synth.normal_f32(992, 3, M)
    q, k, v = (np.zeros(M, np.float32) for _ in range(3))
    assert lib.nf4_ref_gemv_qkv(P(w), P(W_.of(gc, gs)), P(w), bq.ctypes.data, None, None, x.ctypes.data, 1,
                                q.ctypes.data, k.ctypes.data, v.ctypes.data) == 0
    yq, _ = oracle.gemv_qkv([(codes, scales, bq), (gc, gs, None), (codes, scales, None)], x)
    assert np.array_equal(np.concatenate([q, k, v]), yq.astype(np.float32))
    X = synth.normal_bf16(993, 1, 7 * K).reshape(7, K)
    Y = np.zeros((7, M), np.float32)
    assert lib.nf4_ref_gemm_chunk(P(w), X.ctypes.data, 7, Y.ctypes.data) == 0
    assert np.array_equal(Y, oracle.gemm_chunk(codes, scales, X)[0].astype(np.float32))
    ids = np.array([3, 0, 39, 39, 17], np.int64)
    rows32 = np.zeros((5, K), np.float32)
    rows16 = np.zeros((5, K), np.uint16)
    assert lib.nf4_ref_dequant_rows(P(w), ids.ctypes.data, 5, rows32.ctypes.data, 0) == 0
    assert lib.nf4_ref_dequant_rows(P(w), ids.ctypes.data, 5, rows16.ctypes.data, 1) == 0
    f32, b16, bad = oracle.dequant_rows(codes, scales, ids)
    assert bad == 0 and np.array_equal(rows32, f32) and np.array_equal(rows16, b16)
    xr = synth.normal_f32(994, 4, 3 * K).reshape(3, K)
    g = synth.f32_bits_to_bf16((1.0 + 0.25 * synth.normal_f32(994, 5, K)).astype(np.float32))
    yr = np.zeros((3, K), np.float32)
    yb = np.zeros((3, K), np.uint16)
    assert lib.nf4_ref_rmsnorm(xr.ctypes.data, g.ctypes.data, 3, K, ctypes.c_float(1e-6), yr.ctypes.data, 0) == 0
    assert lib.nf4_ref_rmsnorm(xr.ctypes.data, g.ctypes.data, 3, K, ctypes.c_float(1e-6), yb.ctypes.data, 1) == 0
    y64, _ = oracle.rmsnorm(xr, g, float(np.float32(1e-6)))
    assert np.array_equal(yr, y64.astype(np.float32))
    assert np.array_equal(yb, np.array([[oracle.round_bf16(v) for v in row] for row in y64], np.uint16))
    # invalid arguments are refused
    assert lib.nf4_ref_gemv(None, x.ctypes.data, 1, y.ctypes.data) == -1
    assert lib.nf4_ref_gemm_chunk(P(w), X.ctypes.data, 33, Y.ctypes.data) == -1
