"""Helpers for the GPU parity tests: run a layer through the C ABI, compare
with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll

PREC_NAME = {si.PREC_FP32: "fp32", si.PREC_TF32: "tf32", si.PREC_BF16: "bf16"}


def device_inputs(X, W, b, precision):
    dt = torch.bfloat16 if precision == si.PREC_BF16 else torch.float32
    x = torch.from_numpy(np.ascontiguousarray(X)).cuda().to(dt)
    w = torch.from_numpy(np.ascontiguousarray(W)).cuda().to(dt)
    bias = None if b is None else torch.from_numpy(np.ascontiguousarray(b)).cuda()
    return x, w, bias


def run(X, W, b, precision, epilogue=si.EPI_NONE, plan=None, ctx=None):
    """Y (float64 numpy) from the GPU for fp32 host inputs X, W, bias."""
    return run_t(X, W, b, precision, epilogue, plan, ctx).float().cpu().numpy().astype(np.float64)


def run_t(X, W, b, precision, epilogue=si.EPI_NONE, plan=None, ctx=None):
    """Y as a CUDA tensor in the output dtype."""
    x, w, bias = device_inputs(X, W, b, precision)
    epi = "gelu" if epilogue == si.EPI_GELU else "none"
    if plan is None:
        y = tll.forward(x, w, bias, epilogue=epi, precision=PREC_NAME[precision], ctx=ctx)
    else:
        y = tll.forward_plan(plan, x, w, bias, epilogue=epi, precision=PREC_NAME[precision], ctx=ctx)
    torch.cuda.synchronize()
    (ctx or tll.default_context(0)).check()
    return y


def check_layer(layer: si.Layer, plan=None, ctx=None, tol=None):
    """Full-output parity of one layer; returns rel_err."""
    X, W, b = si.make_inputs(layer)
    y = run(X, W, b, layer.precision, layer.epilogue, plan=plan, ctx=ctx)
    ref = oracle.linear(X, W, b, bool(layer.epilogue))
    err = oracle.rel_err(y, ref)
    tol = oracle.TOL[layer.precision] if tol is None else tol
    assert np.all(np.isfinite(y)), f"{layer.name}: non-finite output"
    assert err <= tol, f"{layer.name} plan={plan}: rel_err {err:.3e} > {tol:g}"
    return err


def sample_indices(M, N, count, seed=0):
    """Sampled (m, n) pairs: random ones plus the first/last row and column."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, count))
    ns = list(rng.integers(0, N, count))
    for n in np.linspace(0, N - 1, 64).astype(int):
        ms += [0, M - 1]
        ns += [int(n), int(n)]
    for m in np.linspace(0, M - 1, 64).astype(int):
        ms += [int(m), int(m)]
        ns += [0, N - 1]
    return np.array(ms, np.int64), np.array(ns, np.int64)


def check_layer_sampled(layer: si.Layer, count=2048, plan=None):
    """Large-shape parity on sampled outputs computed one by one by the oracle.
    The scale max|Y_ref| comes from the sampled entries (a lower bound of the
    full max), which makes the test stricter, not looser."""
    X, W, b = si.make_inputs(layer)
    y = run_t(X, W, b, layer.precision, layer.epilogue, plan=plan)
    ms, ns = sample_indices(layer.M, layer.N, count)
    got = y[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].float().cpu().numpy().astype(np.float64)
    ref = oracle.linear_entries(X, W, ms, ns, b, bool(layer.epilogue))
    err = oracle.rel_err(got, ref)
    tol = oracle.TOL[layer.precision]
    assert bool(torch.isfinite(y).all()), f"{layer.name}: non-finite output"
    assert err <= tol, f"{layer.name}: sampled rel_err {err:.3e} > {tol:g}"
    return err
