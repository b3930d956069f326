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
