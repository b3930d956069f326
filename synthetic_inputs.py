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

The pages only require that every version of a kernel is fed from one seeded
generator (a GPT-2-class transformer on a GPU, "Results"); the generator choice is this
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
CHUNK = 1 << 21  # elements per block: arrays are built block by block in reused buffers


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (variant 13) on a uint64 array, wrapping (returns a copy)."""
    z = np.array(z, dtype=np.uint64, copy=True)
    _mix_inplace(z, np.empty_like(z))
    return z


def _mix_inplace(z: np.ndarray, tmp: np.ndarray) -> None:
    np.right_shift(z, np.uint64(30), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)


def stream_base(seed: int, tid: int) -> np.uint64:
    """Start state of tensor stream ``tid`` under ``seed``."""
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + np.uint64(tid + 1) * GAMMA
    return _mix(np.array([s], dtype=np.uint64))[0]


class _Blocks:
    """Reused buffers for block-wise generation (large arrays without large temporaries)."""

    def __init__(self, n):
        self.iota = np.arange(1, n + 1, dtype=np.uint64)
        self.z = np.empty(n, dtype=np.uint64)
        self.t = np.empty(n, dtype=np.uint64)

    def draws(self, base, start, n):
        """Draws start .. start+n-1 of the stream with start state ``base`` (a view of a buffer)."""
        z, t = self.z[:n], self.t[:n]
        np.add(self.iota[:n], np.uint64(start), out=z)
        np.multiply(z, GAMMA, out=z)
        np.add(z, base, out=z)
        _mix_inplace(z, t)
        return z


def draws(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """uint64 draws ``start .. start+count-1`` of stream ``tid``."""
    base = stream_base(seed, tid)
    out = np.empty(count, dtype=np.uint64)
    blk = _Blocks(min(max(count, 1), CHUNK))
    for c0 in range(0, count, CHUNK):
        n = min(CHUNK, count - c0)
        out[c0:c0 + n] = blk.draws(base, start + c0, n)
    return out


def uniform_pm1(seed: int, tid: int, shape) -> np.ndarray:
    """fp32 array uniform on [-1, 1) with 24-bit resolution: u * 2**-23 - 1 for the
    top 24 bits u of each draw (exact in fp32)."""
    count = int(np.prod(shape))
    base = stream_base(seed, tid)
    out = np.empty(count, dtype=np.float32)
    blk = _Blocks(min(max(count, 1), CHUNK))
    for c0 in range(0, count, CHUNK):
        n = min(CHUNK, count - c0)
        z = blk.draws(base, c0, n)
        np.right_shift(z, np.uint64(40), out=z)
        o = out[c0:c0 + n]
        np.copyto(o, z, casting="unsafe")
        np.multiply(o, np.float32(2.0 ** -23), out=o)
        np.subtract(o, np.float32(1.0), out=o)
    return out.reshape(shape)


def normal(seed: int, tid: int, shape, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """fp32 array ~ N(mu, sigma) by Box-Muller from paired draws (2i, 2i+1), in
    float64: mu + sigma * sqrt(-2 ln u1) cos(2 pi u2), u1 in (0, 1], u2 in [0, 1)."""
    count = int(np.prod(shape))
    base = stream_base(seed, tid)
    out = np.empty(count, dtype=np.float32)
    half = max(1, min(count, CHUNK // 2))
    blk = _Blocks(2 * half)
    a = np.empty(half, dtype=np.float64)
    b = np.empty(half, dtype=np.float64)
    two_pi = 2.0 * math.pi
    for c0 in range(0, count, half):
        n = min(half, count - c0)
        z = blk.draws(base, 2 * c0, 2 * n)
        np.right_shift(z, np.uint64(11), out=z)
        u1, u2 = a[:n], b[:n]
        np.copyto(u1, z[0::2], casting="unsafe")
        np.add(u1, 1.0, out=u1)
        np.multiply(u1, 2.0 ** -53, out=u1)
        np.copyto(u2, z[1::2], casting="unsafe")
        np.multiply(u2, 2.0 ** -53, out=u2)
        np.log(u1, out=u1)
        np.multiply(u1, -2.0, out=u1)
        np.sqrt(u1, out=u1)
        np.multiply(u2, two_pi, out=u2)
        np.cos(u2, out=u2)
        np.multiply(u1, u2, out=u1)
        np.multiply(u1, sigma, out=u1)
        np.add(u1, mu, out=u1)
        np.copyto(out[c0:c0 + n], u1, casting="same_kind")
    return out.reshape(shape)


def small_ints(seed: int, tid: int, shape, lo: int = -4, hi: int = 4) -> np.ndarray:
    """fp32 array of integers uniform on [lo, hi]: (draw >> 32) mod (hi - lo + 1) + lo."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    v = (draws(seed, tid, n) >> np.uint64(32)) % span
    return (v.astype(np.int64) + lo).astype(np.float32).reshape(shape)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16; returns the uint16 bit patterns."""
    src = np.ascontiguousarray(a, dtype=np.float32).reshape(-1).view(np.uint32)
    out = np.empty(src.size, dtype=np.uint16)
    m = min(max(src.size, 1), CHUNK)
    r = np.empty(m, dtype=np.uint32)
    for c0 in range(0, src.size, CHUNK):
        n = min(CHUNK, src.size - c0)
        b, rr = src[c0:c0 + n], r[:n]
        np.right_shift(b, np.uint32(16), out=rr)
        np.bitwise_and(rr, np.uint32(1), out=rr)
        np.add(rr, np.uint32(0x7FFF), out=rr)
        np.add(rr, b, out=rr)  # wraps only for NaN/inf inputs, which the recipes never produce
        np.right_shift(rr, np.uint32(16), out=rr)
        np.copyto(out[c0:c0 + n], rr, casting="unsafe")
    return out.reshape(np.shape(a))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(src.shape, dtype=np.uint32)
    np.copyto(out, src, casting="unsafe")
    np.left_shift(out, np.uint32(16), out=out)
    return out.view(np.float32)


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

# The one-row sites ("Optimizing a GPT-2-class transformer on a GPU", Act II:
# only the final token's logits are needed): the LM head at M = 1.
GPT2_LOGITS_M1 = (
    Layer("gpt2_logits_m1_fp32", 1, 50257, 768, PREC_FP32, bias=False),
    Layer("gpt2_logits_m1_bf16", 1, 50257, 768, PREC_BF16, bias=False),
)

ALL_WORKLOADS = ((SQUARE_256_FP32, SKINNY_16x4096, SQUARE_4096_FP32, SQUARE_4096_TF32) + GPT2_M128_FP32 + GPT2_M8192_BF16 +
                 GPT2_LOGITS_M1)


@dataclass(frozen=True)
class Attention:
    """One self-attention problem read from the qkv projection's output:
    B sequences of T tokens, H heads of width D, bf16 q/k/v."""

    name: str
    B: int
    T: int
    H: int
    D: int
    causal: bool = True
    seed: int = 0

    @property
    def C(self) -> int:
        return self.H * self.D

    @property
    def flops(self) -> int:
        """Multiply-adds of q k^T and p v, counted as 2 FLOPs each (the causal
        case visits half of the key-query pairs)."""
        pairs = self.T * (self.T + 1) // 2 if self.causal else self.T * self.T
        return 4 * self.B * self.H * pairs * self.D

    def algorithmic_bytes(self) -> int:
        """q, k, v read and the output written once, bf16."""
        return 2 * (3 * self.B * self.T * self.C + self.B * self.T * self.C)


def make_qkv(att: Attention) -> np.ndarray:
    """The (B*T) x 3C qkv projection output, N(0, 1) rounded to bf16 (fp32
    array of the exact values the GPU receives). Tensor stream id 4."""
    return round_bf16(normal(att.seed, 4, (att.B * att.T, 3 * att.C), 0.0, 1.0))


# GPT-2 small's attention at the batched shape (64 sequences x 128 tokens, 12
# heads of 64), causal, reading the qkv layer's output.
GPT2_ATTN_B64 = Attention("gpt2_attn_b64_t128_bf16", 64, 128, 12, 64, causal=True)
