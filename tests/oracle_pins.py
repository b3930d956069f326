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


# ----------------------------------------------------------------- backward
#
# Backward pins take ``bwd = (dz, dx, dw)``: dz(X, W, b, dY, gelu) -> dZ,
# dx(dZ, W) -> dX, dw(dZ, X) -> (dW, db), and ``gg(z) -> gelu'(z)``; the
# forward ``f`` is the (already pinned) forward oracle.

def _grid(seed, stream, shape, step=2.0 ** -8):
    """Values on a dyadic grid in [-1, 1): X +- 2^-12 stays exact in fp32."""
    return (np.round(si.uniform_pm1(seed, stream, shape) / step) * step).astype(np.float32)


def pin_gelu_grad_function(gg, g):
    """gelu'(0) = 1/2; gelu'(z) + gelu'(-z) = 1 (from g(z) - g(-z) = z); the
    slope tends to 1 and 0 in the tails; it is the central difference of the
    forward GELU; and torch autograd of gelu(approximate="tanh") agrees."""
    assert gg(np.array([0.0]))[0] == 0.5
    z = np.linspace(-6.0, 6.0, 241)
    assert np.max(np.abs(gg(z) + gg(-z) - 1.0)) <= 1e-14
    assert abs(gg(np.array([12.0]))[0] - 1.0) <= 1e-12 and abs(gg(np.array([-12.0]))[0]) <= 1e-12
    h = 1e-5
    fd = (g(z + h) - g(z - h)) / (2 * h)
    assert np.max(np.abs(gg(z) - fd)) <= 1e-8
    t = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(t, approximate="tanh").sum().backward()
    assert np.max(np.abs(gg(z) - t.grad.numpy())) <= 1e-12


def pin_backward_finite_differences(f, bwd):
    """d/dX, d/dW, d/db of L = sum(G * f(X, W, b, act)) by central differences
    of the forward oracle equal dX = dZ W, dW = dZ^T X, db = sum_m dZ with
    dZ = G * act'(Z), for the identity and for GELU."""
    dz, dx, dw = bwd
    M, N, K = 3, 4, 5
    X, W, b, G = _grid(51, 1, (M, K)), _grid(51, 2, (N, K)), _grid(51, 3, (N,)), _grid(51, 4, (M, N))
    h = 2.0 ** -12
    for gelu in (False, True):
        L = lambda X_, W_, b_: float(np.sum(G.astype(np.float64) * f(X_, W_, b_, gelu)))
        dZ = dz(X, W, b, G, gelu)
        dZf = dZ.astype(np.float32)  # the backward GEMMs take fp32 operands
        gx, (gw, gb) = dx(dZf, W), dw(dZf, X)
        num_x, num_w, num_b = np.zeros((M, K)), np.zeros((N, K)), np.zeros(N)
        for idx in np.ndindex(M, K):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            num_x[idx] = (L(Xp, W, b) - L(Xm, W, b)) / (2 * h)
        for idx in np.ndindex(N, K):
            Wp, Wm = W.copy(), W.copy()
            Wp[idx] += h
            Wm[idx] -= h
            num_w[idx] = (L(X, Wp, b) - L(X, Wm, b)) / (2 * h)
        for n in range(N):
            bp, bm = b.copy(), b.copy()
            bp[n] += h
            bm[n] -= h
            num_b[n] = (L(X, W, bp) - L(X, W, bm)) / (2 * h)
        # dZ is rounded to fp32 before the GEMMs: allow that (2^-24 relative)
        for got, num, what in ((gx, num_x, "dX"), (gw, num_w, "dW"), (gb, num_b, "db")):
            assert np.max(np.abs(got - num)) <= 1e-5 * max(1.0, np.max(np.abs(num))), f"{what} gelu={gelu}"


def pin_backward_closed_forms(bwd):
    """Index maps: W = I gives dX = dZ; X = I gives dW = dZ^T; a one-hot dZ at
    (m0, n0) gives dX = W[n0] in row m0 and dW = X[m0] in row n0 (non-square,
    so a transposed map cannot pass); dZ = 1 gives db = M."""
    dz, dx, dw = bwd
    M, N, K = 5, 7, 3
    dZ = _grid(52, 1, (M, N))
    assert np.array_equal(dx(dZ, np.eye(N, dtype=np.float32)), dZ.astype(np.float64))
    dW, _ = dw(dZ, np.eye(M, dtype=np.float32))
    assert np.array_equal(dW, dZ.T.astype(np.float64))
    X, W = _grid(52, 2, (M, K)), _grid(52, 3, (N, K))
    one = np.zeros((M, N), dtype=np.float32)
    one[3, 5] = 1.0
    ex = np.zeros((M, K))
    ex[3] = W[5]
    assert np.array_equal(dx(one, W), ex), "one-hot dX"
    ew = np.zeros((N, K))
    ew[5] = X[3]
    dW, db = dw(one, X)
    assert np.array_equal(dW, ew), "one-hot dW"
    ebias = np.zeros(N)
    ebias[5] = 1.0
    assert np.array_equal(db, ebias), "one-hot db"
    _, db = dw(np.ones((M, N), dtype=np.float32), X)
    assert np.array_equal(db, np.full(N, float(M))), "db of ones"
    # identity activation: dZ = dY exactly
    dY = _grid(52, 4, (M, N))
    assert np.array_equal(dz(X, W, None, dY, False), dY.astype(np.float64))


BACKWARD_PINS = (pin_backward_finite_differences, pin_backward_closed_forms)


# ------------------------------------------- fused residual, LayerNorm fold, dX through GELU


def pin_residual(fr):
    """Y = act(X W^T + b) + R: W = 0 and no bias give Y = R exactly (gelu(0) = 0);
    small integers match a brute-force integer sum exactly; the residual is
    added after the activation (bias-only layer: gelu(b) + R, with GELU from
    torch, not gelu(b + R))."""
    rng = _rng(61)
    M, N, K = 3, 5, 4
    R = rng.integers(-9, 10, (M, N)).astype(np.float32)
    X = rng.integers(-3, 4, (M, K)).astype(np.float32)
    for gelu in (False, True):
        assert np.array_equal(fr(X, np.zeros((N, K), np.float32), R, None, gelu), R.astype(np.float64))
    W = rng.integers(-3, 4, (N, K)).astype(np.float32)
    b = rng.integers(-5, 6, (N,)).astype(np.float32)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            want[m, n] = sum(int(X[m, k]) * int(W[n, k]) for k in range(K)) + int(b[n]) + int(R[m, n])
    assert np.array_equal(fr(X, W, R, b, False), want)
    bias = np.array([1.0, -0.5, 2.0], np.float32)
    Rb = np.full((2, 3), 1.5, np.float32)
    g = torch.nn.functional.gelu(torch.tensor(bias, dtype=torch.float64), approximate="tanh").numpy()
    got = fr(np.zeros((2, 1), np.float32), np.zeros((3, 1), np.float32), Rb, bias, True)
    assert np.max(np.abs(got - (g[None, :] + 1.5))) <= 1e-15


def pin_layernorm(ln):
    """LayerNorm equals torch's layer_norm in float64 (biased variance, eps
    inside the root); xhat has mean 0 and mean square var / (var + eps); with
    eps = 0 it is invariant to x -> a x + c (a > 0)."""
    rng = _rng(62)
    X = (rng.standard_normal((4, 37)) * 3 + 1).astype(np.float32)
    gamma = rng.standard_normal(37).astype(np.float32)
    beta = rng.standard_normal(37).astype(np.float32)
    ref = torch.nn.functional.layer_norm(torch.tensor(X, dtype=torch.float64), (37,),
                                         torch.tensor(gamma, dtype=torch.float64),
                                         torch.tensor(beta, dtype=torch.float64), eps=1e-5).numpy()
    assert np.max(np.abs(ln(X, gamma, beta, 1e-5) - ref)) <= 1e-12
    xh = ln(X, None, None, 1e-5)
    Xd = X.astype(np.float64)
    var = Xd.var(axis=1)
    assert np.max(np.abs(xh.mean(axis=1))) <= 1e-14
    assert np.max(np.abs((xh ** 2).mean(axis=1) - var / (var + 1e-5))) <= 1e-12
    Y = (X * 4.0 + 3.0).astype(np.float32)  # exact in fp32 for these magnitudes? close enough at 1e-6
    assert np.max(np.abs(ln(Y, None, None, 0.0) - ln(X, None, None, 0.0))) <= 1e-5


def pin_fold(fold, ln):
    """The fold is exact algebra: W LN(x) + b = Wf xhat + bf for random data
    (LayerNorm from torch, products by numpy in float64); gamma = 1, beta = 0
    leave W and b unchanged; small integers match a brute-force fold."""
    rng = _rng(63)
    N, K, M = 7, 11, 5  # N != K: a transposed or mis-indexed fold cannot pass
    W = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    gamma = (rng.standard_normal(K) + 1).astype(np.float32)
    beta = rng.standard_normal(K).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float32)
    t = lambda a: torch.tensor(a, dtype=torch.float64)
    lnx = torch.nn.functional.layer_norm(t(X), (K,), t(gamma), t(beta), eps=1e-5).numpy()
    xhat = torch.nn.functional.layer_norm(t(X), (K,), None, None, eps=1e-5).numpy()
    Wf, bf = fold(W, gamma, beta, b)
    want = lnx @ W.astype(np.float64).T + b.astype(np.float64)
    got = xhat @ Wf.T + bf
    assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))
    Wf1, bf1 = fold(W, np.ones(K, np.float32), np.zeros(K, np.float32), b)
    assert np.array_equal(Wf1, W.astype(np.float64)) and np.array_equal(bf1, b.astype(np.float64))
    Wi = rng.integers(-4, 5, (N, K)).astype(np.float32)
    gi = rng.integers(-3, 4, K).astype(np.float32)
    bi = rng.integers(-3, 4, K).astype(np.float32)
    ci = rng.integers(-9, 10, N).astype(np.float32)
    Wf, bf = fold(Wi, gi, bi, ci)
    for n in range(N):
        assert bf[n] == int(ci[n]) + sum(int(Wi[n, k]) * int(bi[k]) for k in range(K))
        for k in range(K):
            assert Wf[n, k] == int(Wi[n, k]) * int(gi[k])
    _, bf0 = fold(Wi, gi, None, None)
    assert np.array_equal(bf0, np.zeros(N))


def pin_dx_gelu(dxg):
    """dX carried through the GELU of the previous layer: the central
    difference of L(Zp) = sum(G * (gelu(Zp) W^T + b)) (GELU from torch, the
    product by numpy, all in float64) equals dxg(G, W, Zp); at Zp = 0 the
    slope is 1/2, so W = I gives G / 2 exactly."""
    M, N, K = 3, 4, 5
    G, W, b, Zp = _grid(64, 1, (M, N)), _grid(64, 2, (N, K)), _grid(64, 3, (N,)), _grid(64, 4, (M, K))
    gelu_t = lambda z: torch.nn.functional.gelu(torch.tensor(z, dtype=torch.float64), approximate="tanh").numpy()
    Wd, bd, Gd = W.astype(np.float64), b.astype(np.float64), G.astype(np.float64)
    L = lambda Z: float(np.sum(Gd * (gelu_t(Z) @ Wd.T + bd)))
    h = 2.0 ** -12
    num = np.zeros((M, K))
    for idx in np.ndindex(M, K):
        Zpp, Zpm = Zp.astype(np.float64).copy(), Zp.astype(np.float64).copy()
        Zpp[idx] += h
        Zpm[idx] -= h
        num[idx] = (L(Zpp) - L(Zpm)) / (2 * h)
    got = dxg(G, W, Zp)
    assert np.max(np.abs(got - num)) <= 1e-6 * max(1.0, np.max(np.abs(num)))
    Gs = _grid(64, 5, (M, K))
    assert np.array_equal(dxg(Gs, np.eye(K, dtype=np.float32), np.zeros((M, K), np.float32)),
                          Gs.astype(np.float64) / 2)


NEXT4_PINS = (pin_residual, pin_layernorm, pin_fold, pin_dx_gelu)


# ------------------------------------------------------------------ self-attention
#
# An attention callable: attn(qkv, B, T, H, D, causal, scale) -> (out, lse) in
# float64, with qkv the (B*T) x 3C projection output (C = H*D; q, k, v at
# column offsets 0, C, 2C, head h at h*D), out (B*T) x C and lse B x H x T.


def _qkv_split(qkv, B, T, H, D):
    """(q, k, v), each B x H x T x D float64, from the projection layout."""
    x = qkv.astype(np.float64).reshape(B, T, 3, H, D)
    return tuple(np.ascontiguousarray(x[:, :, i].transpose(0, 2, 1, 3)) for i in range(3))


def pin_attention_library(attn):
    """Equals torch's scaled_dot_product_attention in float64 (causal and not,
    a non-square shape so that a swapped axis cannot pass, scale 1/sqrt(D) and
    another), and lse equals torch.logsumexp of the scaled, masked scores."""
    rng = _rng(71)
    B, T, H, D = 2, 7, 3, 5
    qkv = rng.standard_normal((B * T, 3 * H * D)).astype(np.float32)
    q, k, v = (torch.tensor(a) for a in _qkv_split(qkv, B, T, H, D))
    for causal in (True, False):
        for scale in (1.0 / math.sqrt(D), 0.37):
            out, lse = attn(qkv, B, T, H, D, causal, scale)
            ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
            ref = ref.permute(0, 2, 1, 3).reshape(B * T, H * D).numpy()
            assert np.max(np.abs(out - ref)) <= 1e-13, (causal, scale)
            s = (q @ k.transpose(-1, -2)) * scale
            if causal:
                s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
            assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-13, (causal, scale)


def pin_attention_uniform(attn):
    """q = 0: every visible key scores 0, so a query's output is the mean of
    the visible values (the prefix mean when causal) and lse is the log of
    their count."""
    rng = _rng(72)
    B, T, H, D = 1, 6, 2, 3
    qkv = rng.standard_normal((B * T, 3 * H * D)).astype(np.float32)
    qkv[:, : H * D] = 0.0
    _, _, v = _qkv_split(qkv, B, T, H, D)
    for causal in (True, False):
        out, lse = attn(qkv, B, T, H, D, causal, 0.5)
        for h in range(H):
            for i in range(T):
                n = i + 1 if causal else T
                want = v[0, h, :n].mean(axis=0)
                assert np.max(np.abs(out[i, h * D:(h + 1) * D] - want)) <= 1e-15, (causal, h, i)
                assert abs(lse[0, h, i] - math.log(n)) <= 1e-15


def pin_attention_one_hot(attn):
    """Orthogonal keys and queries that each point at one visible key with a
    large score: the softmax picks that key and the output is its value (the
    rest weigh e^-40 of it); causal queries point at key i // 2, full ones at
    key T - 1 - i (a non-involutive choice, so a transposed index fails)."""
    B, T, H, D = 1, 6, 1, 6
    rng = _rng(73)
    v = rng.standard_normal((T, D)).astype(np.float32)
    for causal in (True, False):
        pick = [i // 2 if causal else (2 * i + 1) % T for i in range(T)]
        qkv = np.zeros((T, 3 * D), np.float32)
        qkv[np.arange(T), np.array(pick)] = 40.0          # q_i = 40 e_pick(i)
        qkv[np.arange(T), D + np.arange(T)] = 1.0          # k_j = e_j
        qkv[:, 2 * D:] = v
        out, _ = attn(qkv, B, T, H, D, causal, 1.0)
        assert np.max(np.abs(out - v[pick].astype(np.float64))) <= 1e-14, causal


def pin_attention_key_order(attn):
    """Full (non-causal) attention does not depend on the order of the keys:
    permuting the k and v rows together (q fixed) leaves every output."""
    rng = _rng(74)
    B, T, H, D = 1, 9, 2, 4
    qkv = rng.standard_normal((B * T, 3 * H * D)).astype(np.float32)
    perm = (np.arange(T) * 4 + 1) % T
    shuffled = qkv.copy()
    shuffled[:, H * D:] = qkv[perm, H * D:]
    a, la = attn(qkv, B, T, H, D, False, 0.5)
    b, lb = attn(shuffled, B, T, H, D, False, 0.5)
    assert np.max(np.abs(a - b)) <= 1e-14 and np.max(np.abs(la - lb)) <= 1e-14


ATTENTION_PINS = (pin_attention_library, pin_attention_uniform, pin_attention_one_hot, pin_attention_key_order)
