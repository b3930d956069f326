"""Backward (training) GEMMs against the oracle: dX = dZ W, dW = dZ^T X,
db = column sums of dZ, and dZ = dY * gelu'(Z)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll
from gpu_util import PREC_NAME

pytestmark = pytest.mark.gpu

FP32, TF32, BF16 = si.PREC_FP32, si.PREC_TF32, si.PREC_BF16


@pytest.fixture(scope="module", autouse=True)
def _early_start_all():
    """Back-to-back library calls only: the programmatic early start is safe
    here and is what the back-to-back tests exercise (the default is off)."""
    c = tll.default_context(0)
    c.set_option(tll.OPT_EARLY_START, tll.EARLY_ALL)
    yield
    c.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)


def _dt(precision):
    return torch.bfloat16 if precision == BF16 else torch.float32


def _dev(a, precision):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(_dt(precision)).cuda()


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def _inputs(M, N, K, precision, seed, ints=False):
    if ints:
        dZ = si.small_ints(seed, 1, (M, N))
        W = si.small_ints(seed, 2, (N, K))
        X = si.small_ints(seed, 3, (M, K))
    else:
        dZ = si.normal(seed, 1, (M, N), 0.0, 0.1)
        W = si.normal(seed, 2, (N, K), 0.0, 0.02)
        X = si.normal(seed, 3, (M, K))
    if precision == BF16:
        dZ, W, X = si.round_bf16(dZ), si.round_bf16(W), si.round_bf16(X)
    return dZ.astype(np.float32), W.astype(np.float32), X.astype(np.float32)


def _tol(precision):
    # TF32 backward runs exact fp32 FFMAs
    return oracle.TOL[BF16] if precision == BF16 else oracle.TOL[FP32]


SHAPES = [(257, 136, 200), (128, 768, 768), (384, 3072, 768), (64, 768, 3072), (1, 8, 8), (5, 16, 24)]


@pytest.mark.parametrize("precision", [FP32, TF32, BF16])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_backward_data_and_weight(precision, M, N, K):
    dZ, W, X = _inputs(M, N, K, precision, seed=M + N + K)
    dz, w, x = _dev(dZ, precision), _dev(W, precision), _dev(X, precision)
    dx = tll.backward_data(dz, w, precision=PREC_NAME[precision])
    dw, db = tll.backward_weight(dz, x, db=True, precision=PREC_NAME[precision])
    torch.cuda.synchronize()
    tll.default_context(0).check()
    ref_dx = oracle.backward_dx(dZ, W)
    ref_dw, ref_db = oracle.backward_dw(dZ, X)
    assert oracle.rel_err(_host(dx), ref_dx) <= _tol(precision), "dX"
    assert oracle.rel_err(_host(dw), ref_dw) <= _tol(precision), "dW"
    assert oracle.rel_err(db.double().cpu().numpy(), ref_db) <= oracle.TOL[FP32], "db"
    # bitwise repeatable
    dx2 = tll.backward_data(dz, w, precision=PREC_NAME[precision])
    dw2, db2 = tll.backward_weight(dz, x, db=True, precision=PREC_NAME[precision])
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2) and torch.equal(db, db2)


@pytest.mark.parametrize("precision", [FP32, BF16])
def test_backward_small_integers_exact(precision):
    """Integer operands: every product and partial sum is exact, so the GPU
    equals the oracle bit for bit (bf16 results: the oracle rounded to bf16).
    A wrong index map of either transpose case cannot pass."""
    M, N, K = 192, 264, 320
    dZ, W, X = _inputs(M, N, K, precision, seed=5, ints=True)
    dz, w, x = _dev(dZ, precision), _dev(W, precision), _dev(X, precision)
    dx = tll.backward_data(dz, w, precision=PREC_NAME[precision])
    dw, db = tll.backward_weight(dz, x, db=True, precision=PREC_NAME[precision])
    torch.cuda.synchronize()
    ref_dx = oracle.backward_dx(dZ, W)
    ref_dw, ref_db = oracle.backward_dw(dZ, X)
    if precision == BF16:
        ref_dx = si.round_bf16(ref_dx.astype(np.float32)).astype(np.float64)
        ref_dw = si.round_bf16(ref_dw.astype(np.float32)).astype(np.float64)
    assert np.array_equal(_host(dx), ref_dx)
    assert np.array_equal(_host(dw), ref_dw)
    assert np.array_equal(db.double().cpu().numpy(), ref_db)


@pytest.mark.parametrize("precision", [FP32, BF16])
def test_gelu_backward(precision):
    M, N = 37, 1000
    dY = si.normal(8, 1, (M, N))
    Z = si.normal(8, 2, (M, N), 0.0, 2.0)
    if precision == BF16:
        dY, Z = si.round_bf16(dY), si.round_bf16(Z)
    dy, z = _dev(dY, precision), _dev(Z, precision)
    dz = tll.gelu_backward(dy, z, precision=PREC_NAME[precision])
    torch.cuda.synchronize()
    ref = oracle.gelu_backward(dY, Z)
    assert oracle.rel_err(_host(dz), ref) <= (oracle.TOL[BF16] if precision == BF16 else oracle.TOL[FP32])
    # in place
    tll.gelu_backward(dy, z, out=dy, precision=PREC_NAME[precision])
    torch.cuda.synchronize()
    assert torch.equal(dy, dz)


def test_backward_zero_sizes():
    for precision in (FP32, BF16):
        dt = _dt(precision)
        dz = torch.zeros((4, 0), device="cuda", dtype=dt)
        w = torch.zeros((0, 8), device="cuda", dtype=dt)
        dx = torch.full((4, 8), 7.0, device="cuda", dtype=dt)
        tll.backward_data(dz, w, out=dx, precision=PREC_NAME[precision])
        x = torch.ones((0, 8), device="cuda", dtype=dt)
        dz2 = torch.zeros((0, 16), device="cuda", dtype=dt)
        dw = torch.full((16, 8), 7.0, device="cuda", dtype=dt)
        db = torch.full((16,), 7.0, device="cuda")
        tll.backward_weight(dz2, x, out=dw, db=db, precision=PREC_NAME[precision])
        torch.cuda.synchronize()
        assert bool((dx == 0).all()) and bool((dw == 0).all()) and bool((db == 0).all())


def test_backward_status_codes():
    ctx = tll.default_context(0)
    lib = tll.library()
    s = torch.cuda.current_stream().cuda_stream
    dz = torch.zeros((16, 12), device="cuda", dtype=torch.bfloat16)  # N = 12: bf16 rows not 16-byte aligned
    w = torch.zeros((12, 64), device="cuda", dtype=torch.bfloat16)
    dx = torch.zeros((16, 64), device="cuda", dtype=torch.bfloat16)
    assert lib.lin_backward_data(ctx._h, 16, 12, 64, dz.data_ptr(), w.data_ptr(), dx.data_ptr(), 2, s) == tll.ERR_ALIGN
    dzf = torch.zeros((16, 12), device="cuda")
    wf = torch.zeros((12, 64), device="cuda")
    dxf = torch.zeros((16, 64), device="cuda")
    assert lib.lin_backward_data(ctx._h, 16, 12, 64, dzf.data_ptr(), wf.data_ptr(), dzf.data_ptr(), 0, s) == tll.ERR_ARG
    assert lib.lin_backward_data(ctx._h, 16, 12, 64, dzf.data_ptr(), wf.data_ptr(), dxf.data_ptr(), 0, s) == tll.OK
    assert lib.lin_backward_data(ctx._h, -1, 12, 64, dzf.data_ptr(), wf.data_ptr(), dxf.data_ptr(), 0, s) == tll.ERR_ARG
    small = tll.Context(0, workspace_bytes=4096)
    x = torch.zeros((1024, 64), device="cuda")
    dz2 = torch.zeros((1024, 512), device="cuda")
    dw = torch.zeros((512, 64), device="cuda")
    db = torch.zeros((512,), device="cuda")
    assert lib.lin_backward_weight(small._h, 1024, 512, 64, dz2.data_ptr(), x.data_ptr(), dw.data_ptr(),
                                   db.data_ptr(), 0, s) == tll.ERR_WORKSPACE
    torch.cuda.synchronize()
    ctx.check()
    small.close()


@pytest.mark.parametrize("precision", [FP32, BF16])
def test_training_step_through_the_layer(precision):
    """Forward with GELU (saving Z = X W^T + b with a second forward call),
    then dZ = dY * gelu'(Z), dX and dW, db: each against the oracle on the
    GPU's own inputs of that step; and the chain against the oracle's dZ."""
    M, N, K = 256, 1024, 768
    X = si.normal(21, 1, (M, K))
    W = si.normal(21, 2, (N, K), 0.0, 0.02)
    b = si.normal(21, 3, (N,), 0.0, 0.02)
    dY = si.normal(21, 4, (M, N), 0.0, 0.1)
    if precision == BF16:
        X, W, dY = si.round_bf16(X), si.round_bf16(W), si.round_bf16(dY)
    x, w, dy = _dev(X, precision), _dev(W, precision), _dev(dY, precision)
    bias = torch.from_numpy(b).cuda()
    prec = PREC_NAME[precision]
    z = tll.forward(x, w, bias, epilogue="none", precision=prec)
    dz = tll.gelu_backward(dy, z, precision=prec)
    dx = tll.backward_data(dz, w, precision=prec)
    dw, db = tll.backward_weight(dz, x, db=True, precision=prec)
    torch.cuda.synchronize()
    tol = _tol(precision)
    dZg = dz.float().cpu().numpy()
    assert oracle.rel_err(_host(dx), oracle.backward_dx(dZg, W)) <= tol
    ref_dw, ref_db = oracle.backward_dw(dZg, X)
    assert oracle.rel_err(_host(dw), ref_dw) <= tol
    assert oracle.rel_err(db.double().cpu().numpy(), ref_db) <= oracle.TOL[FP32]
    # the whole chain against the oracle's own dZ (its Z in double)
    ref_dz = oracle.backward_dz(X, W, dY, b, True)
    assert oracle.rel_err(_host(dz), ref_dz) <= (2e-2 if precision == BF16 else 1e-4)


@pytest.mark.parametrize("M,N,K", [(8192, 3072, 768), (8192, 768, 3072)], ids=["fc1", "fc2"])
def test_backward_gpt2_m8192_bf16_full(M, N, K):
    """The batched GPT-2 fc1 and fc2 layers' backward at full size, every
    output of dX, dW and db against the oracle."""
    dZ, W, X = _inputs(M, N, K, BF16, seed=99)
    dz, w, x = _dev(dZ, BF16), _dev(W, BF16), _dev(X, BF16)
    dx = tll.backward_data(dz, w)
    dw, db = tll.backward_weight(dz, x, db=True)
    torch.cuda.synchronize()
    ref_dw, ref_db = oracle.backward_dw(dZ, X)
    assert oracle.rel_err(_host(dx), oracle.backward_dx(dZ, W)) <= oracle.TOL[BF16]
    assert oracle.rel_err(_host(dw), ref_dw) <= oracle.TOL[BF16]
    assert oracle.rel_err(db.double().cpu().numpy(), ref_db) <= oracle.TOL[FP32]


@pytest.mark.parametrize("precision", [FP32, BF16])
def test_backward_back_to_back(precision):
    """Backward calls launched back to back (early start; fp32 split-K shares
    the workspace): independent calls into separate outputs equal the same
    calls made one at a time."""
    M, N, K = 128, 3072, 768
    dZ, W, X = _inputs(M, N, K, precision, seed=77)
    dzs = [_dev(dZ * (1 + i), precision) for i in range(3)]
    w, x = _dev(W, precision), _dev(X, precision)
    prec = PREC_NAME[precision]
    outs = []
    for i in range(6):
        outs.append(tll.backward_data(dzs[i % 3], w, precision=prec))
        outs.append(tll.backward_weight(dzs[i % 3], x, db=True, precision=prec))
    torch.cuda.synchronize()
    for i in range(6):
        ref_dx = tll.backward_data(dzs[i % 3], w, precision=prec)
        torch.cuda.synchronize()
        ref_dw, ref_db = tll.backward_weight(dzs[i % 3], x, db=True, precision=prec)
        torch.cuda.synchronize()
        assert torch.equal(outs[2 * i], ref_dx), i
        assert torch.equal(outs[2 * i + 1][0], ref_dw) and torch.equal(outs[2 * i + 1][1], ref_db), i
    tll.default_context(0).check()


def test_backward_weight_k_split():
    """A weight gradient with few output tiles and a long reduction, called
    on a fresh stream (nothing to overlap with): the tensor cores split the
    reduction and add the splits in order. Every output against the oracle,
    and bitwise repeatable."""
    M, N, K = 8192, 768, 256
    dZ, _, X = _inputs(M, N, K, BF16, seed=123)
    dz, x = _dev(dZ, BF16), _dev(X, BF16)
    outs = []
    for _ in range(2):
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            outs.append(tll.backward_weight(dz, x, db=True, stream=st))
        st.synchronize()
    dw, db = outs[0]
    assert torch.equal(dw, outs[1][0]) and torch.equal(db, outs[1][1])
    ref_dw, ref_db = oracle.backward_dw(dZ, X)
    assert oracle.rel_err(_host(dw), ref_dw) <= oracle.TOL[BF16]
    assert oracle.rel_err(db.double().cpu().numpy(), ref_db) <= oracle.TOL[FP32]
