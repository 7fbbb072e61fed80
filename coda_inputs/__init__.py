"""Seeded synthetic inputs for the CODA GEMM-epilogue workloads.

This module is the only code shared by the CUDA path's tests/bench and the
oracle. It draws random tensors and encodes them as bfloat16 bit patterns; it
holds none of the method's arithmetic (no GEMM, normalisation, activation,
rotation or loss).

Recipe (the same for every workload):
  * ``numpy.random.Generator(PCG64)`` seeded from ``SeedSequence(seed)``;
    ``seed`` defaults to 0. One ``spawn`` child per tensor, in the order the
    workload lists its tensors, so a forward tensor is identical whether or not
    the backward tensors are requested.
  * Draw float32 standard normals, scale (and shift) in float32, then round
    to bfloat16 with round-to-nearest-even. The result is returned as
    ``uint16`` bit patterns so every consumer reads the same bytes.
  * Labels are int32, uniform in ``[0, V)``.

Distributions (weights ~ N(0, 1/fan_in), activations ~ N(0, 1),
gamma ~ 1 + 0.1 N(0, 1)) follow the workload statements that accompany the
CODA paper's kernel table (GEMM+RoPE QKV projection, GEMM+SwiGLU up-projection,
GEMM-RMSNorm-GEMM, LM-head GEMM + cross-entropy).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "f32_to_bf16_bits",
    "normal_bf16",
    "f32_to_e4m3_bits",
    "normal_e4m3",
    "fp8_problem",
    "rms_chain",
    "rope_problem",
    "swiglu_problem",
    "ce_problem",
    "block_problem",
    "BLOCK_SIZES",
    "WORKLOADS",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return uint16 bits.

    Inputs here are finite normals, so NaN/Inf handling is not needed; it is
    still guarded so a NaN stays a NaN.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def f32_to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to FP8 E4M3 (1 sign bit, 4 exponent bits with bias
    7, 3 mantissa bits, no infinities; 0x7F/0xFF are NaN) with round-to-nearest-
    even, saturating finite magnitudes above 448 (the largest finite value) to
    448. Returns uint8 bit patterns.

    The rounding is done in float64, where every step is exact: a magnitude
    below 2^-6 is a multiple of 2^-9 (subnormal), otherwise 2^e (1 + m/8)."""
    x = np.asarray(a, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    ax = np.minimum(np.abs(x), 448.0)
    mant, exp = np.frexp(ax)            # ax = mant * 2^exp, mant in [0.5, 1)
    e = exp - 1                         # ax = 2^e * (2 mant)
    normal = ax >= 2.0 ** -6
    # normal: (e + 7) * 8 + rint(8 * (2 mant - 1)); a carry out of the mantissa
    # (rint gives 8) lands in the exponent field, as it should
    code_n = (e + 7) * 8 + np.rint(16.0 * mant - 8.0)
    # subnormal: multiples of 2^-9; rint gives 0..8, and 8 is the smallest normal (0x08)
    code_s = np.rint(ax * 512.0)
    code = np.where(normal, code_n, code_s)
    code = np.minimum(code, 0x7E).astype(np.uint8)
    out = code | sign
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint8(0x7F)
    return out


def _children(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """bf16 bits of ``mean + std * N(0, 1)`` drawn in float32."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return f32_to_bf16_bits(x)


def normal_e4m3(rng: np.random.Generator, shape) -> np.ndarray:
    """E4M3 bits of N(0, 1) drawn in float32 (the tensor's value is a per-tensor
    scale times these)."""
    return f32_to_e4m3_bits(rng.standard_normal(size=shape, dtype=np.float32))


def fp8_problem(M: int, K: int, N: int, seed: int = 0, labels: bool = False) -> dict:
    """FP8 (E4M3) GEMM operands with per-tensor scales, for the FP8 mainloop:
    A[M,K] = sA * e4m3(N(0,1)) with sA = 1 (activations), and the weight stored
    K-major as B[N,K] = sB * e4m3(N(0,1)) with sB = 1/sqrt(K), so that the
    weight is distributed as N(0, 1/K) like the bf16 workloads' and the product
    is O(1). Returns the bit arrays and the float scales; with labels=True also
    int32 labels uniform in [0, N) (the cross-entropy workload).
    Tensors in spawn order: A, B, labels."""
    g = _children(seed, 3)
    out = {"A": normal_e4m3(g[0], (M, K)), "B": normal_e4m3(g[1], (N, K)),
           "sA": 1.0, "sB": float(1.0 / np.sqrt(K))}
    if labels:
        out["labels"] = g[2].integers(0, N, size=(M,), dtype=np.int32)
    return out


def rms_chain(M: int, K: int, d: int, N2: int, seed: int = 0, bwd_K: int | None = None) -> dict:
    """GEMM -> residual add -> RMSNorm -> GEMM problem.

    Tensors, in spawn order: x[M,K] ~ N(0,1), W0[K,d] ~ N(0,1/K),
    z[M,d] ~ N(0,1), gamma[d] ~ 1 + 0.1 N(0,1), W1[d,N2] ~ N(0,1/d), and for
    the backward stand-in GEMM that produces the output gradient dY = dO Wn:
    dO[M,bwd_K] ~ N(0,1), Wn[bwd_K,N2] ~ N(0,1/bwd_K).
    """
    g = _children(seed, 7)
    out = {
        "x": normal_bf16(g[0], (M, K)),
        "W0": normal_bf16(g[1], (K, d), std=1.0 / np.sqrt(K)),
        "z": normal_bf16(g[2], (M, d)),
        "gamma": normal_bf16(g[3], (d,), std=0.1, mean=1.0),
        "W1": normal_bf16(g[4], (d, N2), std=1.0 / np.sqrt(d)),
    }
    if bwd_K is not None:
        out["dO"] = normal_bf16(g[5], (M, bwd_K))
        out["Wn"] = normal_bf16(g[6], (bwd_K, N2), std=1.0 / np.sqrt(bwd_K))
    return out


def rms_chain_outliers(M: int, K: int, d: int, N2: int, seed: int = 0, frac: float = 0.01,
                       scale: float = 20.0) -> dict:
    """The rms_chain problem with outlier channels in the residual stream: a
    `frac` share of the d channels of z (chosen by the seed) is drawn `scale`
    times wider, a synthetic stand-in for the few large-magnitude channels of
    trained models' residual streams. Same spawn order as rms_chain, plus one
    child for the channel choice."""
    g = _children(seed, 8)
    z = g[2].standard_normal(size=(M, d), dtype=np.float32)
    cols = g[7].choice(d, size=max(1, int(round(frac * d))), replace=False)
    z[:, cols] *= np.float32(scale)
    return {
        "x": normal_bf16(g[0], (M, K)),
        "W0": normal_bf16(g[1], (K, d), std=1.0 / np.sqrt(K)),
        "z": f32_to_bf16_bits(z),
        "gamma": normal_bf16(g[3], (d,), std=0.1, mean=1.0),
        "W1": normal_bf16(g[4], (d, N2), std=1.0 / np.sqrt(d)),
        "outlier_cols": np.sort(cols),
    }


def rope_problem(M: int, K: int, N3: int, seed: int = 0, with_bwd: bool = True) -> dict:
    """QKV projection X[M,K] ~ N(0,1) times W[K,N3] ~ N(0,1/K).

    Backward stand-in operands of the same shapes: A[M,K] ~ N(0,1),
    B[K,N3] ~ N(0,1/K) (their product plays the gradient of the rotated
    output).
    """
    g = _children(seed, 4)
    out = {
        "X": normal_bf16(g[0], (M, K)),
        "W": normal_bf16(g[1], (K, N3), std=1.0 / np.sqrt(K)),
    }
    if with_bwd:
        out["A"] = normal_bf16(g[2], (M, K))
        out["B"] = normal_bf16(g[3], (K, N3), std=1.0 / np.sqrt(K))
    return out


def swiglu_problem(M: int, K: int, F: int, seed: int = 0, with_bwd: bool = True) -> dict:
    """MLP up-projection X[M,K] ~ N(0,1) times gate/up-interleaved Wgu[K,2F] ~ N(0,1/K).

    Backward: dY[M,K] ~ N(0,1) (gradient of the down-projection output) and the
    down-projection weight Wd[F,K] ~ N(0,1/F), stored [F, K].
    """
    g = _children(seed, 4)
    out = {
        "X": normal_bf16(g[0], (M, K)),
        "Wgu": normal_bf16(g[1], (K, 2 * F), std=1.0 / np.sqrt(K)),
    }
    if with_bwd:
        out["dY"] = normal_bf16(g[2], (M, K))
        out["Wd"] = normal_bf16(g[3], (F, K), std=1.0 / np.sqrt(F))
    return out


def ce_problem(M: int, K: int, V: int, seed: int = 0) -> dict:
    """LM head H[M,K] ~ N(0,1) times W[K,V] ~ N(0,1/K); labels int32 uniform in [0,V)."""
    g = _children(seed, 3)
    return {
        "H": normal_bf16(g[0], (M, K)),
        "W": normal_bf16(g[1], (K, V), std=1.0 / np.sqrt(K)),
        "labels": g[2].integers(0, V, size=(M,), dtype=np.int32),
    }


def block_problem(M: int, d: int, F: int, seed: int = 0, with_bwd: bool = True) -> dict:
    """One period of the block-level chain: two GEMM-residual-RMSNorm-GEMM
    structures (RoPE path, then SwiGLU path).

    Tensors, in spawn order:
      P[M,F] ~ N(0,1)        activation entering the down projection
      Wd[F,d] ~ N(0,1/F)     down projection
      x[M,d] ~ N(0,1)        residual stream entering the block
      gamma1[d] ~ 1 + 0.1 N(0,1)
      Wqkv[d,3d] ~ N(0,1/d)  QKV projection
      O[M,d] ~ N(0,1)        attention-core output (the attention core itself is not part of the chain)
      Wo[d,d] ~ N(0,1/d)     attention output projection
      gamma2[d] ~ 1 + 0.1 N(0,1)
      Wgu[d,2F] ~ N(0,1/d)   gate/up projection, gate and up columns interleaved
    and for the backward:
      dQKV[M,3d] ~ N(0,1)    gradient of the rotated QKV (from the attention backward)
      gh[M,d] ~ N(0,1)       gradient of the next period's residual output
      Wdn[F,d] ~ N(0,1/F)    the next period's down projection
    """
    g = _children(seed, 12)
    out = {
        "P": normal_bf16(g[0], (M, F)),
        "Wd": normal_bf16(g[1], (F, d), std=1.0 / np.sqrt(F)),
        "x": normal_bf16(g[2], (M, d)),
        "gamma1": normal_bf16(g[3], (d,), std=0.1, mean=1.0),
        "Wqkv": normal_bf16(g[4], (d, 3 * d), std=1.0 / np.sqrt(d)),
        "O": normal_bf16(g[5], (M, d)),
        "Wo": normal_bf16(g[6], (d, d), std=1.0 / np.sqrt(d)),
        "gamma2": normal_bf16(g[7], (d,), std=0.1, mean=1.0),
        "Wgu": normal_bf16(g[8], (d, 2 * F), std=1.0 / np.sqrt(d)),
    }
    if with_bwd:
        out["dQKV"] = normal_bf16(g[9], (M, 3 * d))
        out["gh"] = normal_bf16(g[10], (M, d))
        out["Wdn"] = normal_bf16(g[11], (F, d), std=1.0 / np.sqrt(F))
    return out


# Block-level chain sizes: 16K tokens at the hidden widths of the 1B, 7B and
# 70B model scales; F and head_dim as in Llama-3-family models of those widths;
# positions = row mod 4096 (four 4096-token sequences).
BLOCK_SIZES = {
    2048: dict(M=16384, d=2048, F=8192, head_dim=64),
    4096: dict(M=16384, d=4096, F=14336, head_dim=128),
    8192: dict(M=16384, d=8192, F=28672, head_dim=128),
}

# The five workloads, by name, with their full sizes.
WORKLOADS = {
    "rmsnorm_chain_tiny": dict(kind="rms_chain", M=256, K=512, d=512, N2=512, eps=1e-6),
    "rope_qkv_4096": dict(kind="rope", M=4096, K=4096, N3=12288, head_dim=128, theta=10000.0,
                          S=4096, rope_cols=8192),
    "swiglu_up_4096": dict(kind="swiglu", M=4096, K=4096, F=14336),
    "rmsnorm_chain_8192": dict(kind="rms_chain", M=8192, K=8192, d=8192, N2=8192, eps=1e-6,
                               bwd_K=8192),
    "lm_head_ce_8192": dict(kind="ce", M=8192, K=4096, V=32768),
}
# FP8 (E4M3) mainloop variants of the single-GEMM forward operators, same shapes
# as their bf16 workloads; weights stored K-major ([N, K]).
WORKLOADS["fp8_rope_qkv_4096"] = dict(kind="fp8_rope", M=4096, K=4096, N=12288, head_dim=128, theta=10000.0,
                                      S=4096, rope_cols=8192)
WORKLOADS["fp8_swiglu_up_4096"] = dict(kind="fp8_swiglu", M=4096, K=4096, N=28672)
WORKLOADS["fp8_lm_head_ce_8192"] = dict(kind="fp8_ce", M=8192, K=4096, N=32768)
for _d, _b in BLOCK_SIZES.items():
    WORKLOADS[f"block_d{_d}"] = dict(kind="block", S=4096, theta=10000.0, eps=1e-6, rope_cols=2 * _d, **_b)
