"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module draws random numbers and rounds them to the storage types; it holds
none of the method's arithmetic (no codebook, no quantization, no products).
Every tensor comes from its own numpy ``Generator(PCG64(seed * 1000 + tensor_id))``
stream, drawn in float64 and rounded once to fp32 (round to nearest even), and
for bf16 tensors rounded again from that fp32 to bf16 (nearest even).  Weights
are drawn row-block by row-block from one stream, which yields the same values
as a single draw.

The five workloads mirror the projections of the Qwen2.5-3B / 14B-shaped models
that "Decode V2 -- resident executor" times (section 6 "Linear primitive" table,
section 10 "Qwen2.5-3B"), with synthetic N(0, 0.02) weights in place of trained
checkpoints.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SEED_STRIDE = 1000
W_STD = 0.02


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed * SEED_STRIDE + tensor_id))


def f32_bits_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_f32(seed: int, tensor_id: int, n: int, std: float = 1.0) -> np.ndarray:
    z = rng(seed, tensor_id).standard_normal(n)
    return (std * z).astype(np.float32)


def token_ids(seed: int, tensor_id: int, n: int, vocab: int) -> np.ndarray:
    """n token ids drawn uniformly from [0, vocab), int64."""
    return rng(seed, tensor_id).integers(0, vocab, n, dtype=np.int64)


def weights(seed: int, tensor_id: int, M: int, K: int, std: float = W_STD,
            rows_per_draw: int = 4096) -> np.ndarray:
    """fp32 [M, K] weights ~ N(0, std^2), drawn in row blocks from one stream."""
    g = rng(seed, tensor_id)
    out = np.empty((M, K), np.float32)
    for r0 in range(0, M, rows_per_draw):
        r1 = min(M, r0 + rows_per_draw)
        out[r0:r1] = (std * g.standard_normal((r1 - r0) * K)).astype(np.float32).reshape(r1 - r0, K)
    return out


def normal_bf16(seed: int, tensor_id: int, n: int) -> np.ndarray:
    return f32_bits_to_bf16(normal_f32(seed, tensor_id, n))


def silu_product_bf16(seed: int, tid_a: int, tid_b: int, n: int) -> np.ndarray:
    """bf16 activation drawn as silu(z1) * z2 with z1, z2 ~ N(0, 1), float64 then rounded.

    This is the input recipe of a down projection's activation (the output of a
    SwiGLU layer), not the method's epilogue.
    """
    z1 = rng(seed, tid_a).standard_normal(n)
    z2 = rng(seed, tid_b).standard_normal(n)
    v = z1 / (1.0 + np.exp(-z1)) * z2
    return f32_bits_to_bf16(v.astype(np.float32))


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "gemv", "residual", "swiglu", "argmax", "chunk", "qkv", "embed", "glu", "rmsnorm"
    M: int
    K: int
    N: int
    seed: int
    x_dtype: str  # "f32" or "bf16"
    description: str
    M_kv: int = 0  # qkv: rows of k and of v (M is q's rows)


WORKLOADS = {
    "tiny": Workload("tiny", "gemv", 256, 512, 1, 0, "f32",
                     "tiny NF4 GEMV 256x512, x fp32 N(0,1), fp32 out"),
    "down_residual": Workload("down_residual", "residual", 2048, 11008, 1, 1, "bf16",
                              "3B down_proj 2048x11008, x bf16 silu(z1)*z2, + fp32 residual"),
    "swiglu": Workload("swiglu", "swiglu", 11008, 2048, 1, 2, "bf16",
                       "3B gate/up 2x 11008x2048, x bf16 N(0,1), bf16 silu(g)*u out"),
    "glu3b": Workload("glu3b", "glu", 11008, 2048, 1, 2, "bf16",
                      "3B gate/up (the swiglu weights) interleaved into one 22016x2048 matrix, row 2c gate c, "
                      "row 2c+1 up c, x bf16 N(0,1), bf16 silu(g)*u out"),
    "lm_head_argmax": Workload("lm_head_argmax", "argmax", 151936, 2048, 1, 3, "bf16",
                               "3B lm_head 151936x2048, x bf16 N(0,1), fp32 logits + argmax"),
    "chunk14b": Workload("chunk14b", "chunk", 13824, 5120, 32, 4, "bf16",
                         "14B-shaped 13824x5120, X 32x5120 bf16 N(0,1), Y fp32 [32][13824]"),
    "gemv14b": Workload("gemv14b", "gemv", 13824, 5120, 1, 4, "bf16",
                        "14B-shaped 13824x5120 at N=1, x = X[0] of the chunk workload"),
    "qkv3b": Workload("qkv3b", "qkv", 2048, 2048, 1, 5, "bf16",
                      "3B q/k/v 2048x2048 + 2x 256x2048 in one launch, x bf16 N(0,1), fp32 biases N(0,1)",
                      M_kv=256),
    "embed_prefill": Workload("embed_prefill", "embed", 151936, 2048, 4096, 6, "bf16",
                              "3B embedding table 151936x2048 kept as NF4, 4096 token ids uniform, bf16 rows out"),
    "rmsnorm3b": Workload("rmsnorm3b", "rmsnorm", 1, 2048, 1, 7, "bf16",
                          "3B decode RMSNorm: x fp32 [2048] N(0,1), bf16 gain 1 + 0.25 N(0,1), eps 1e-6, bf16 out"),
    "rmsnorm_chunk14b": Workload("rmsnorm_chunk14b", "rmsnorm", 32, 5120, 32, 8, "bf16",
                                 "14B prefill-chunk RMSNorm: x fp32 [32][5120] N(0,1), bf16 gain, eps 1e-6, "
                                 "bf16 out"),
}


def workload_inputs(w: Workload, M: int | None = None) -> dict:
    """fp32 weights and activations for a workload (optionally only its first M rows).

    Keys: ``W`` (and ``Wu`` for swiglu) fp32 [M, K]; ``x`` (fp32 or bf16 bits);
    ``r`` fp32 residual; ``X`` bf16 bits [N, K] for the chunk.
    """
    M = w.M if M is None else M
    K = w.K
    s = w.seed
    d = {}
    if w.kind == "embed":
        d["W"] = weights(s, 0, M, K)
        d["ids"] = token_ids(s, 1, w.N, M)
    elif w.kind == "qkv":
        d["W"] = weights(s, 0, M, K)
        d["Wk"] = weights(s, 1, w.M_kv, K)
        d["Wv"] = weights(s, 2, w.M_kv, K)
        d["x"] = normal_bf16(s, 3, K)
        d["bq"] = normal_f32(s, 4, M)
        d["bk"] = normal_f32(s, 5, w.M_kv)
        d["bv"] = normal_f32(s, 6, w.M_kv)
    elif w.kind == "swiglu":
        d["W"] = weights(s, 0, M, K)
        d["Wu"] = weights(s, 1, M, K)
        d["x"] = normal_bf16(s, 2, K)
    elif w.kind == "glu":  # M outputs: 2 M rows, gate and up alternating
        d["W"] = np.empty((2 * M, K), np.float32)
        d["W"][0::2] = weights(s, 0, M, K)
        d["W"][1::2] = weights(s, 1, M, K)
        d["x"] = normal_bf16(s, 2, K)
    elif w.kind == "residual":
        d["W"] = weights(s, 0, M, K)
        d["x"] = silu_product_bf16(s, 1, 2, K)
        d["r"] = normal_f32(s, 3, M)
    elif w.kind == "rmsnorm":  # M rows of K
        d["x"] = normal_f32(s, 0, M * K).reshape(M, K)
        d["w"] = f32_bits_to_bf16((1.0 + 0.25 * normal_f32(s, 1, K)).astype(np.float32))
    elif w.kind in ("chunk",) or w.name == "gemv14b":
        d["W"] = weights(s, 0, M, K)
        X = normal_bf16(s, 1, 32 * K).reshape(32, K)
        d["X"] = X[: w.N] if w.kind == "chunk" else X[:1]
        d["x"] = X[0].copy()
    else:
        d["W"] = weights(s, 0, M, K)
        d["x"] = normal_f32(s, 1, K) if w.x_dtype == "f32" else normal_bf16(s, 1, K)
    return d
