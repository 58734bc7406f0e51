"""Seeded synthetic inputs for the groupwise low-bit linear layer.

This module is the one thing the CPU oracle and the CUDA path share: it only
draws random numbers and rounds them to the storage formats (bf16, fp16,
uint8 codes).  It holds none of the layer's arithmetic (no packing, no
dequantisation, no products).

Value recipe (the decode workloads the pages measure use Llama-3.x layer
shapes; trained weights are not needed to exercise the kernels, so values
are synthetic):

* x      = bf16_rn(N(0, 1)); optionally ceil(1% of K) distinct columns are
           multiplied by 20 before rounding (outlier columns).
* codes  = uniform integers in [0, 2^b - 1], one per byte.
* scale  = fp16_rn(U[1e-3, 1e-2]).
* zero   = fp16_rn(-scale_fp16 * U[6, 9]).
* bias   = fp16_rn(N(0, 0.02)).

Every tensor draws from its own stream, keyed by (seed, tensor id, shape,
bits, group), so the same call always yields the same bytes.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# Stream ids per tensor.
STREAM_X, STREAM_CODES, STREAM_SCALE, STREAM_ZERO_U, STREAM_BIAS, STREAM_OUTLIER = 1, 2, 3, 4, 5, 6
STREAM_WEIGHT = 7


def rng(seed: int, stream: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, *key])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def f16_bits(a: np.ndarray) -> np.ndarray:
    """Round to fp16 (nearest even, numpy's conversion); returns uint16 bit patterns."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


@dataclasses.dataclass
class Layer:
    """Host copies of one layer's inputs.  fp16/bf16 tensors are uint16 bit patterns."""
    M: int
    K: int
    N: int
    bits: int
    group: int
    x: np.ndarray           # [M, K] bf16 bits
    codes: np.ndarray       # [N, K] uint8, one code per byte
    scales: np.ndarray      # [N, K/g] fp16 bits
    zeros: np.ndarray       # [N, K/g] fp16 bits
    bias: np.ndarray | None  # [N] fp16 bits or None


def make_x(seed: int, M: int, K: int, outliers: bool = False, key: tuple = ()) -> np.ndarray:
    x = rng(seed, STREAM_X, M, K, *key).standard_normal((M, K), dtype=np.float32)
    if outliers and K > 0:
        n_out = int(np.ceil(0.01 * K))
        cols = rng(seed, STREAM_OUTLIER, K, *key).permutation(K)[:n_out]
        x[:, cols] *= 20.0
    return f32_to_bf16_bits(x)


def make_codes(seed: int, N: int, K: int, bits: int, key: tuple = ()) -> np.ndarray:
    return rng(seed, STREAM_CODES, N, K, bits, *key).integers(
        0, 1 << bits, size=(N, K), dtype=np.uint8)


def make_scale_zero(seed: int, N: int, G: int, key: tuple = ()):
    s = f16_bits(rng(seed, STREAM_SCALE, N, G, *key).uniform(1e-3, 1e-2, size=(N, G)))
    u = rng(seed, STREAM_ZERO_U, N, G, *key).uniform(6.0, 9.0, size=(N, G))
    s64 = s.view(np.float16).astype(np.float64)
    z = f16_bits(-s64 * u)
    return s, z


def make_bias(seed: int, N: int, key: tuple = ()) -> np.ndarray:
    return f16_bits(rng(seed, STREAM_BIAS, N, *key).normal(0.0, 0.02, size=N))


def make_weights(seed: int, N: int, K: int, key: tuple = ()) -> np.ndarray:
    """Float weights [N, K] (float32) for the quantiser: N(0, 0.02), with one
    row in 64 scaled by 8 and ceil(1% of K) columns by 4, so that groups span a
    wide range of magnitudes."""
    r = rng(seed, STREAM_WEIGHT, N, K, *key)
    w = r.normal(0.0, 0.02, size=(N, K)).astype(np.float32)
    if N > 0 and K > 0:
        w[r.permutation(N)[: max(1, N // 64)]] *= 8.0
        w[:, r.permutation(K)[: int(np.ceil(0.01 * K))]] *= 4.0
    return w


def make_layer(seed: int, M: int, K: int, N: int, bits: int, group: int,
               bias: bool = False, outliers: bool = False) -> Layer:
    key = (bits, group)
    scales, zeros = make_scale_zero(seed, N, K // group, (K, bits, group))
    return Layer(
        M=M, K=K, N=N, bits=bits, group=group,
        x=make_x(seed, M, K, outliers, key),
        codes=make_codes(seed, N, K, bits, key),
        scales=scales, zeros=zeros,
        bias=make_bias(seed, N, key) if bias else None,
    )


# ---------------------------------------------------------------------------
# Workloads: Llama-3.x decode/prefill linear-layer shapes (K, N).
# ---------------------------------------------------------------------------
LLAMA_8B = {"qkv": (4096, 6144), "o": (4096, 4096), "gate_up": (4096, 28672), "down": (14336, 4096)}
LLAMA_3B = {"qkv": (3072, 5120), "o": (3072, 3072), "gate_up": (3072, 16384), "down": (8192, 3072)}
LLAMA_1B = {"qkv": (2048, 3072), "o": (2048, 2048), "gate_up": (2048, 16384), "down": (8192, 2048)}

# Small single layer: M=1, K=N=4096, b=4, g=64, no bias, seed 0.
SINGLE_QMV = dict(M=1, K=4096, N=4096, bits=4, group=64, bias=False, outliers=False)
