"""Pins for the CPU oracle: facts the mathematics fixes, independent of it.

Each ``pin_*`` takes a linear-layer callable ``f(X, W, bias, gelu) -> Y``
(float64) and raises AssertionError when the callable breaks the fact. The
pins are chosen so that a plausible mistake anywhere in the oracle fails at
least one of them: a transposed W, a wrong row/column index, a dropped or
misplaced bias, a wrong activation constant, a low-precision accumulator, a
dropped term. ``tests/test_oracle_pins.py`` runs them on the oracle and on
mutants that plant each of those mistakes.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def pin_identity(f):
    """W = I: Y = X exactly, for several K."""
    for K, M in ((1, 3), (7, 5), (64, 4), (130, 2)):
        X = si.uniform_pm1(11, K, (M, K))
        Y = f(X, np.eye(K, dtype=np.float32), None, False)
        assert Y.shape == (M, K)
        assert np.array_equal(Y, X.astype(np.float64)), f"identity K={K}"


def pin_permutation(f):
    """W[n, p(n)] = 1 for a non-involutive permutation p: Y[:, n] = X[:, p(n)]."""
    K = 37
    p = (np.arange(K) * 5 + 3) % K  # affine map on Z_37, not its own inverse
    assert not np.array_equal(p[p], np.arange(K))
    W = np.zeros((K, K), dtype=np.float32)
    W[np.arange(K), p] = 1.0
    X = si.uniform_pm1(12, 0, (6, K))
    Y = f(X, W, None, False)
    assert np.array_equal(Y, X[:, p].astype(np.float64)), "permutation"


def pin_selector_rect(f):
    """Non-square selector: N=11 outputs, K=29 inputs, W[n, (3n+2) mod K] = 1."""
    N, K, M = 11, 29, 5
    sel = (3 * np.arange(N) + 2) % K
    W = np.zeros((N, K), dtype=np.float32)
    W[np.arange(N), sel] = 1.0
    X = si.uniform_pm1(13, 0, (M, K))
    Y = f(X, W, None, False)
    assert Y.shape == (M, N)
    assert np.array_equal(Y, X[:, sel].astype(np.float64)), "rectangular selector"


def pin_small_ints(f):
    """Integer inputs in [-4, 4]: every product and partial sum is an exact integer."""
    for (M, N, K) in ((9, 13, 1024), (3, 2, 5), (17, 33, 257)):
        X = si.small_ints(21, M, (M, K))
        W = si.small_ints(22, N, (N, K))
        b = si.small_ints(23, K, (N,))
        exact = X.astype(np.int64) @ W.astype(np.int64).T  # integer matmul, exact
        Y = f(X, W, b, False)
        assert np.array_equal(Y, (exact + b.astype(np.int64)).astype(np.float64)), f"ints {M}x{N}x{K}"


def pin_bruteforce_fsum(f):
    """Tiny shapes with tails: within the double-accumulation error bound of the
    exactly rounded sum (math.fsum of exact fp32 x fp32 products)."""
    eps = 2.0 ** -53
    for M in (1, 2, 5):
        for N in (1, 3, 8):
            for K in (1, 2, 7, 8, 33):
                X = si.normal(31, M * 100 + K, (M, K))
                W = si.normal(32, N * 100 + K, (N, K), 0.0, 0.5)
                b = si.normal(33, N, (N,), 0.0, 0.1)
                Y = f(X, W, b, False)
                for m in range(M):
                    for n in range(N):
                        terms = [float(X[m, k]) * float(W[n, k]) for k in range(K)] + [float(b[n])]
                        exact = math.fsum(terms)
                        bound = (K + 1) * eps * sum(abs(t) for t in terms) + 1e-300
                        assert abs(Y[m, n] - exact) <= bound, (M, N, K, m, n)


def pin_numpy_f64(f):
    """Against numpy's float64 matmul (an independent library reduction)."""
    X = si.normal(41, 0, (24, 300))
    W = si.normal(41, 1, (40, 300), 0.0, 0.02)
    b = si.normal(41, 2, (40,), 0.0, 0.02)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    Y = f(X, W, b, False)
    assert np.max(np.abs(Y - ref)) <= 1e-13 * np.max(np.abs(ref)), "vs numpy float64"


def pin_bias_only(f):
    """X = 0: Y is the bias broadcast over rows (and GELU of it when enabled)."""
    M, N, K = 4, 6, 9
    b = si.normal(51, 0, (N,), 0.0, 1.0)
    Y = f(np.zeros((M, K), np.float32), si.normal(51, 1, (N, K)), b, False)
    assert np.array_equal(Y, np.broadcast_to(b.astype(np.float64), (M, N))), "bias broadcast"
    Yg = f(np.zeros((M, K), np.float32), si.normal(51, 1, (N, K)), b, True)
    ref = torch.nn.functional.gelu(torch.from_numpy(b.astype(np.float64)), approximate="tanh").numpy()
    assert np.allclose(Yg, np.broadcast_to(ref, (M, N)), rtol=1e-14, atol=1e-16), "gelu(bias)"


def pin_empty_k(f):
    """K = 0: the sum is empty, Y = act(bias)."""
    b = np.array([0.5, -2.0, 0.0], np.float32)
    Y = f(np.zeros((2, 0), np.float32), np.zeros((3, 0), np.float32), b, False)
    assert np.array_equal(Y, np.broadcast_to(b.astype(np.float64), (2, 3)))


def pin_bias_then_gelu(f):
    """GELU applies to (sum + bias): integer sums make the pre-activation exact."""
    X = np.array([[1, 2, -1], [0, 3, 1]], np.float32)
    W = np.array([[1, 0, 1], [2, 1, 0], [-1, -1, 1], [0, 0, 2]], np.float32)
    b = np.array([0.5, -3.0, 1.0, -0.25], np.float32)
    pre = X.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    ref = torch.nn.functional.gelu(torch.from_numpy(pre), approximate="tanh").numpy()
    Y = f(X, W, b, True)
    assert np.allclose(Y, ref, rtol=1e-14, atol=1e-16), "gelu(sum + bias)"


def pin_gelu_function(g):
    """The activation alone, g(x) on float64 arrays."""
    x = np.linspace(-12.0, 12.0, 4801)
    y = g(x)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.max(np.abs(y - ref)) <= 1e-14, "vs torch tanh-GELU"
    assert g(np.array([0.0]))[0] == 0.0
    # exact identity of the tanh form: g(x) - g(-x) = x
    assert np.max(np.abs(g(x) - g(-x) - x)) <= 1e-14
    # tails: -> x for large x, -> 0 for very negative x
    assert abs(g(np.array([30.0]))[0] - 30.0) <= 1e-12
    assert abs(g(np.array([-30.0]))[0]) <= 1e-12
    # closeness to the exact GELU x*Phi(x), which the tanh form approximates
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    assert np.max(np.abs(y - exact)) <= 1e-3


def pin_golden_hand_example(f):
    """The hand-worked example in tests/golden/hand_example.txt, exactly."""
    vals = {}
    with open(os.path.join(GOLDEN, "hand_example.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(v) for v in rest]
    M, N, K = int(vals["M"][0]), int(vals["N"][0]), int(vals["K"][0])
    X = np.array(vals["X"], np.float32).reshape(M, K)
    W = np.array(vals["W"], np.float32).reshape(N, K)
    b = np.array(vals["bias"], np.float32)
    Y = f(X, W, b, False)
    assert np.array_equal(Y, np.array(vals["Y"]).reshape(M, N)), "hand example"


LINEAR_PINS = (
    pin_identity, pin_permutation, pin_selector_rect, pin_small_ints, pin_bruteforce_fsum,
    pin_numpy_f64, pin_bias_only, pin_empty_k, pin_bias_then_gelu, pin_golden_hand_example,
)
