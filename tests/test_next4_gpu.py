"""Fused residual epilogue, dX carried through the previous GELU, and the
LayerNorm fold, through the C ABI against the oracle.

The residual runs in every kernel family: each plan of the tuner's menu is
installed for the call signature (lin_set_plan_override) and the call goes
through lin_forward_residual."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll
from transformer_linear_layer_gb300 import autotune
from gpu_util import PREC_NAME

pytestmark = pytest.mark.gpu

BF16, TF32, FP32 = si.PREC_BF16, si.PREC_TF32, si.PREC_FP32


@pytest.fixture(scope="module")
def ctx():
    c = tll.Context(0)
    yield c
    c.close()


def _dev(a, precision):
    dt = torch.bfloat16 if precision == BF16 else torch.float32
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dt)


def _round_out(a, precision):
    """Host array rounded to the output type (the residual the GPU receives)."""
    return si.round_bf16(a.astype(np.float32)) if precision == BF16 else a.astype(np.float32)


def _round_bf16_from_double(a):
    """Round-to-nearest-even of float64 values to bf16 (8 significant bits)."""
    m, e = np.frexp(np.asarray(a, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


@pytest.mark.parametrize("precision,M,N,K", [
    (BF16, 5, 1000, 520), (BF16, 1, 2304, 768), (BF16, 200, 300, 4104), (TF32, 130, 520, 2200),
    (FP32, 130, 520, 2200), (FP32, 3, 500, 256), (BF16, 16, 4096, 768)])
@pytest.mark.parametrize("epi", [si.EPI_NONE, si.EPI_GELU])
def test_residual_every_plan(ctx, precision, M, N, K, epi):
    """Y = act(X W^T + b) + R on every kernel family that runs the shape,
    against the oracle; in place (Y = R) gives the same bits."""
    layer = si.Layer("resid", M, N, K, precision, epi, bias=True)
    X, W, b = si.make_inputs(layer)
    R = _round_out(si.normal(7, 9, (M, N)), precision)
    ref = oracle.linear_residual(X, W, R, b, bool(epi))
    x, w, r = _dev(X, precision), _dev(W, precision), _dev(R, precision)
    bias = torch.from_numpy(b).cuda()
    pname, ename = PREC_NAME[precision], ("gelu" if epi else "none")
    plans = [None] + autotune.candidates(ctx.sm_count, M, N, K, pname, ctx.workspace_bytes)
    kinds = set()
    try:
        for plan in plans:
            ctx.set_override(M, N, K, pname, ename, plan)
            y = tll.forward_residual(x, w, r, bias, epilogue=ename, precision=pname, ctx=ctx)
            kinds.add(ctx.last_plan().kernel)
            inplace = r.clone()
            tll.forward_residual(x, w, inplace, bias, epilogue=ename, precision=pname, out=inplace, ctx=ctx)
            torch.cuda.synchronize()
            ctx.check()
            got = y.double().cpu().numpy()
            assert oracle.rel_err(got, ref) <= oracle.TOL[precision], plan
            assert torch.equal(y, inplace), plan
    finally:
        ctx.set_override(M, N, K, pname, ename, None)
    assert kinds >= {p.kernel for p in plans[1:]}


@pytest.mark.parametrize("precision", [BF16, FP32])
def test_residual_exact_on_integers(ctx, precision):
    """Small integers: X W^T + b + R is exact in fp32 accumulators and in the
    bf16 result (|Y| < 256), so the GPU matches a brute-force sum bit for bit."""
    M, N, K = 130, 136, 72
    X = si.small_ints(3, 1, (M, K), -2, 2)
    W = si.small_ints(3, 2, (N, K), -2, 2)
    b = si.small_ints(3, 3, (N,), -4, 4)
    R = si.small_ints(3, 4, (M, N), -8, 8)
    want = X.astype(np.float64) @ W.astype(np.float64).T + b + R
    assert np.max(np.abs(want)) < 256
    y = tll.forward_residual(_dev(X, precision), _dev(W, precision), _dev(R, precision),
                             torch.from_numpy(b).cuda(), precision=PREC_NAME[precision], ctx=ctx)
    torch.cuda.synchronize()
    assert np.array_equal(y.double().cpu().numpy(), want)


def test_residual_k_zero_and_argument_errors(ctx):
    M, N = 4, 40
    R = torch.randn(M, N, device="cuda")
    b = torch.randn(N, device="cuda")
    x = torch.empty(M, 0, device="cuda")
    w = torch.empty(N, 0, device="cuda")
    y = tll.forward_residual(x, w, R, b, precision="fp32", ctx=ctx)
    torch.cuda.synchronize()
    assert torch.equal(y, b[None, :] + R)
    lib = tll.library()
    Y = torch.empty(M, N, device="cuda")
    xx, ww = torch.randn(M, 64, device="cuda"), torch.randn(N, 64, device="cuda")
    args = (ctx.handle, M, N, 64, ctypes.c_void_p(xx.data_ptr()), ctypes.c_void_p(ww.data_ptr()), None)
    # no residual
    assert lib.lin_forward_residual(*args, None, ctypes.c_void_p(Y.data_ptr()), 0, 0, None) == tll.ERR_ARG
    # a residual that overlaps Y without being Y
    big = torch.empty(M * N + 1, device="cuda")
    rc = lib.lin_forward_residual(*args, ctypes.c_void_p(big.data_ptr() + 4), ctypes.c_void_p(big.data_ptr()), 0, 0,
                                  None)
    assert rc == tll.ERR_ARG


def test_residual_block_in_place_back_to_back(ctx):
    """A GPT-2 block's two residual adds, x = x + proj(a) and x = x + fc2(h),
    in place, back to back on one stream at M = 256 bf16, against the oracle."""
    M, d = 256, 768
    x0 = _round_out(si.normal(11, 1, (M, d)), BF16)
    a = _round_out(si.normal(11, 2, (M, d)), BF16)
    h = _round_out(si.normal(11, 3, (M, 4 * d)), BF16)
    Wp = si.round_bf16(si.normal(11, 4, (d, d), 0.0, 0.02))
    W2 = si.round_bf16(si.normal(11, 5, (d, 4 * d), 0.0, 0.02))
    bp, b2 = si.normal(11, 6, (d,), 0.0, 0.02), si.normal(11, 7, (d,), 0.0, 0.02)
    x = _dev(x0, BF16)
    tll.forward_residual(_dev(a, BF16), _dev(Wp, BF16), x, torch.from_numpy(bp).cuda(), precision="bf16", out=x,
                         ctx=ctx)
    x1 = x.clone()
    tll.forward_residual(_dev(h, BF16), _dev(W2, BF16), x, torch.from_numpy(b2).cuda(), precision="bf16", out=x,
                         ctx=ctx)
    torch.cuda.synchronize()
    ctx.check()
    ref1 = oracle.linear_residual(a, Wp, x0, bp)
    assert oracle.rel_err(x1.double().cpu().numpy(), ref1) <= oracle.TOL[BF16]
    ref2 = oracle.linear_residual(h, W2, x1.float().cpu().numpy(), b2)
    assert oracle.rel_err(x.double().cpu().numpy(), ref2) <= oracle.TOL[BF16]


@pytest.mark.parametrize("precision,M,N,K", [
    (BF16, 256, 768, 3072), (BF16, 200, 136, 520), (FP32, 128, 768, 3072), (FP32, 130, 520, 136),
    (TF32, 64, 200, 72)])
def test_backward_data_gelu(ctx, precision, M, N, K):
    """dZp = (dZ W) * gelu'(Zp) in one pass, against the oracle; in place over
    Zp; for fp32 the same bits as lin_backward_data then lin_gelu_backward."""
    dZ = _round_out(si.normal(21, 1, (M, N), 0.0, 0.1), precision)
    W = _round_out(si.normal(21, 2, (N, K), 0.0, 0.05), precision)
    Zp = _round_out(si.normal(21, 3, (M, K)), precision)
    ref = oracle.backward_dx_gelu(dZ, W, Zp)
    dz, w, zp = _dev(dZ, precision), _dev(W, precision), _dev(Zp, precision)
    pname = PREC_NAME[precision]
    got = tll.backward_data_gelu(dz, w, zp, precision=pname, ctx=ctx)
    inplace = zp.clone()
    tll.backward_data_gelu(dz, w, inplace, out=inplace, precision=pname, ctx=ctx)
    torch.cuda.synchronize()
    ctx.check()
    tol = oracle.TOL[BF16] if precision == BF16 else oracle.TOL[FP32]
    assert oracle.rel_err(got.double().cpu().numpy(), ref) <= tol
    assert torch.equal(got, inplace)
    if precision != BF16:
        two = tll.gelu_backward(tll.backward_data(dz, w, precision=pname, ctx=ctx), zp, precision=pname, ctx=ctx)
        torch.cuda.synchronize()
        assert torch.equal(got, two)


@pytest.mark.parametrize("precision", [FP32, BF16])
@pytest.mark.parametrize("N,K", [(768, 768), (3072, 768), (77, 520)])
def test_fold_layernorm(ctx, precision, N, K):
    """W_out and bias_out equal the oracle's double fold rounded once (bit
    for bit), and the folded layer on xhat matches LN then the layer."""
    W = si.normal(31, 1, (N, K), 0.0, 0.02)
    b = si.normal(31, 2, (N,), 0.0, 0.02)
    gamma = si.normal(31, 3, (K,), 1.0, 0.1)
    beta = si.normal(31, 4, (K,), 0.0, 0.1)
    Wf, bf = oracle.fold_layernorm(W, gamma, beta, b)
    w = torch.from_numpy(W).cuda()
    w_out, b_out = tll.fold_layernorm(w, torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(),
                                      torch.from_numpy(b).cuda(), precision=PREC_NAME[precision], ctx=ctx)
    torch.cuda.synchronize()
    want_w = _round_bf16_from_double(Wf) if precision == BF16 else Wf.astype(np.float32).astype(np.float64)
    assert np.array_equal(w_out.double().cpu().numpy(), want_w)
    assert np.array_equal(b_out.cpu().numpy(), bf.astype(np.float32))
    M = 64
    X = si.normal(31, 5, (M, K), 0.5, 2.0)
    xhat = _round_out(oracle.layernorm(X, None, None, 1e-5), precision)
    ref = oracle.linear(oracle.layernorm(X, gamma, beta, 1e-5).astype(np.float32), W, b)
    y = tll.forward(_dev(xhat, precision), w_out, b_out, precision=PREC_NAME[precision], ctx=ctx)
    torch.cuda.synchronize()
    assert oracle.rel_err(y.double().cpu().numpy(), ref) <= oracle.TOL[precision]
    if precision == FP32:  # in place: W and bias overwritten by their folds
        w2, bb = w.clone(), torch.from_numpy(b).cuda()
        tll.fold_layernorm(w2, torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(), bb,
                           precision="fp32", w_out=w2, bias_out=bb, ctx=ctx)
        torch.cuda.synchronize()
        assert torch.equal(w2, w_out) and torch.equal(bb, b_out)
