"""Seeded synthetic inputs for the linear layer Y = X . W^T (+bias, +GELU).

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It holds input recipes only: a counter-based random number
generator, value distributions, bf16 rounding of inputs, and the workload
shapes. It holds none of the multiply, bias or activation arithmetic.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): state advances by the golden-ratio increment
0x9E3779B97F4A7C15 and each state is passed through the variant-13 finaliser.
Element ``i`` of tensor stream ``tid`` under seed ``seed`` is the output of
that finaliser at ``base(seed, tid) + (i + 1) * gamma`` (wrapping 64-bit), so
any element can be produced without producing the ones before it.

Distributions
-------------
* uniform[-1, 1): the top 24 bits ``u`` of a draw give ``u * 2**-23 - 1``,
  exactly representable in fp32.
* normal(mu, sigma): Box-Muller on two draws (indices 2i, 2i+1) in float64,
  ``sqrt(-2 ln u1) * cos(2 pi u2)``, scaled, then rounded to fp32 (and, for
  bf16 tensors, rounded to nearest-even bf16).

The pages fix only "the same seeded generator" for every version of a kernel
(a GPT-2-class transformer on a GPU, "Results"); the generator choice is this
project's reading, and parity does not depend on it because the oracle and the
GPU receive the identical arrays.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (variant 13) on a uint64 array, wrapping."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def stream_base(seed: int, tid: int) -> np.uint64:
    """Start state of tensor stream ``tid`` under ``seed``."""
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + np.uint64(tid + 1) * GAMMA
    return _mix(np.array([s], dtype=np.uint64))[0]


def draws(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """uint64 draws ``start .. start+count-1`` of stream ``tid``."""
    base = stream_base(seed, tid)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def uniform_pm1(seed: int, tid: int, shape) -> np.ndarray:
    """fp32 array uniform on [-1, 1) with 24-bit resolution."""
    n = int(np.prod(shape))
    u = (draws(seed, tid, n) >> np.uint64(40)).astype(np.float64)
    return (u * 2.0 ** -23 - 1.0).astype(np.float32).reshape(shape)


def normal(seed: int, tid: int, shape, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """fp32 array ~ N(mu, sigma) by Box-Muller from paired draws."""
    n = int(np.prod(shape))
    d = draws(seed, tid, 2 * n)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53  # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return (mu + sigma * z).astype(np.float32).reshape(shape)


def small_ints(seed: int, tid: int, shape, lo: int = -4, hi: int = 4) -> np.ndarray:
    """fp32 array of integers uniform on [lo, hi]."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    v = (draws(seed, tid, n) >> np.uint64(32)) % span
    return (v.astype(np.int64) + lo).astype(np.float32).reshape(shape)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16; returns the uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 values after a round trip through bf16 (nearest-even)."""
    return bf16_bits_to_f32(to_bf16_bits(a))


# ---------------------------------------------------------------------------
# Workloads. Shapes and distributions of the linear layers the pages measure:
# the M=16, 4096x4096 layer ("One multiply, one RTX 5090, eight kernels",
# "The multiply"), GPT-2-small's d=768 layer GEMMs at sequence 128 (the GPT-2
# class transformer page, "Results"), batched 64 x 128 tokens ("Act IV"), and
# the 4096^3 square sgemm ("Writing a CUDA matmul that catches cuBLAS").
# ---------------------------------------------------------------------------

PREC_FP32, PREC_TF32, PREC_BF16 = 0, 1, 2
EPI_NONE, EPI_GELU = 0, 1


@dataclass(frozen=True)
class Layer:
    """One linear-layer problem: shapes, precision, epilogue, input recipe."""

    name: str
    M: int
    N: int
    K: int
    precision: int
    epilogue: int = EPI_NONE
    bias: bool = False
    x_dist: str = "normal"  # "normal" N(0,1) | "uniform" U[-1,1) | "ints"
    w_sigma: float = 0.02  # for w normal; ignored for uniform / ints
    seed: int = 0
    tags: tuple = field(default=())

    @property
    def in_bf16(self) -> bool:
        return self.precision == PREC_BF16

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """X + W + Y once each in their dtypes, plus the fp32 bias."""
        e_in = 2 if self.in_bf16 else 4
        e_out = 2 if self.in_bf16 else 4
        b = e_in * (self.M * self.K + self.N * self.K) + e_out * self.M * self.N
        if self.bias:
            b += 4 * self.N
        return b


def make_inputs(layer: Layer):
    """Host arrays (X, W, bias) for ``layer``.

    X and W are fp32 arrays holding the exact values the GPU receives: for
    bf16 layers they are already rounded to bf16 (use :func:`to_bf16_bits`
    for the device copy). ``bias`` is fp32 or None.
    Tensor stream ids: X = 1, W = 2, bias = 3.
    """
    s = layer.seed
    if layer.x_dist == "uniform":
        X = uniform_pm1(s, 1, (layer.M, layer.K))
        W = uniform_pm1(s, 2, (layer.N, layer.K))
    elif layer.x_dist == "ints":
        X = small_ints(s, 1, (layer.M, layer.K))
        W = small_ints(s, 2, (layer.N, layer.K))
    else:
        X = normal(s, 1, (layer.M, layer.K), 0.0, 1.0)
        W = normal(s, 2, (layer.N, layer.K), 0.0, layer.w_sigma)
    bias = None
    if layer.bias:
        bias = small_ints(s, 3, (layer.N,)) if layer.x_dist == "ints" else normal(s, 3, (layer.N,), 0.0, 0.02)
    if layer.in_bf16:
        X = round_bf16(X)
        W = round_bf16(W)
    return X, W, bias


# The five workloads (sizes and distributions as the pages give them).
SQUARE_256_FP32 = Layer("fp32_256cubed", 256, 256, 256, PREC_FP32, x_dist="uniform")
SKINNY_16x4096 = Layer("skinny_m16_k4096_n4096_bf16", 16, 4096, 4096, PREC_BF16, bias=True)
SQUARE_4096_FP32 = Layer("fp32_4096cubed", 4096, 4096, 4096, PREC_FP32, x_dist="uniform")
SQUARE_4096_TF32 = Layer("tf32_4096cubed", 4096, 4096, 4096, PREC_TF32, x_dist="uniform")
GPT2_M128_FP32 = (
    Layer("gpt2_qkv_m128_fp32", 128, 2304, 768, PREC_FP32, bias=True),
    Layer("gpt2_proj_m128_fp32", 128, 768, 768, PREC_FP32, bias=True),
    Layer("gpt2_fc1_m128_fp32", 128, 3072, 768, PREC_FP32, EPI_GELU, bias=True),
    Layer("gpt2_fc2_m128_fp32", 128, 768, 3072, PREC_FP32, bias=True),
)
GPT2_M8192_BF16 = (
    Layer("gpt2_qkv_m8192_bf16", 8192, 2304, 768, PREC_BF16, bias=True),
    Layer("gpt2_proj_m8192_bf16", 8192, 768, 768, PREC_BF16, bias=True),
    Layer("gpt2_fc1_m8192_bf16", 8192, 3072, 768, PREC_BF16, EPI_GELU, bias=True),
    Layer("gpt2_fc2_m8192_bf16", 8192, 768, 3072, PREC_BF16, bias=True),
    Layer("gpt2_lmhead_m8192_bf16", 8192, 50257, 768, PREC_BF16, bias=False),
)

ALL_WORKLOADS = (SQUARE_256_FP32, SKINNY_16x4096, SQUARE_4096_FP32, SQUARE_4096_TF32) + GPT2_M128_FP32 + GPT2_M8192_BF16
