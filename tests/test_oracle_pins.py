"""The oracle against facts fixed by the mathematics (CPU only).

Also plants mistakes in copies of the oracle (mutants, pure numpy) and checks
that the pins catch every one, and calibrates the acceptance metric the way
the sgemm page does: reordered fp32 summation lands near 1e-6, a real bug
(a misplaced tile) near 1e-1 ("Writing a CUDA matmul that catches cuBLAS",
section "The measurement was nearly wrong").
"""
import math

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from oracle_pins import LINEAR_PINS, pin_gelu_function


def real(X, W, b, gelu):
    return oracle.linear(X, W, b, gelu)


@pytest.mark.parametrize("pin", LINEAR_PINS, ids=lambda p: p.__name__)
def test_oracle_meets_pin(pin):
    pin(real)


def test_gelu_meets_pin():
    pin_gelu_function(oracle.gelu)


def test_entries_match_full():
    X = si.normal(7, 1, (33, 129))
    W = si.normal(7, 2, (71, 129), 0.0, 0.02)
    b = si.normal(7, 3, (71,), 0.0, 0.02)
    full = oracle.linear(X, W, b, True)
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, 33, 500), rng.integers(0, 71, 500)
    assert np.array_equal(oracle.linear_entries(X, W, ms, ns, b, True), full[ms, ns])


def test_thread_count_invariance():
    X = si.normal(8, 1, (16, 1000))
    W = si.normal(8, 2, (50, 1000), 0.0, 0.02)
    assert np.array_equal(oracle.linear(X, W, nthreads=1), oracle.linear(X, W, nthreads=0))


# ---------------------------------------------------------------- mutants ---

def _gelu_np(s, c1=math.sqrt(2.0 / math.pi), c3=0.044715, half=0.5):
    return half * s * (1.0 + np.tanh(c1 * (s + c3 * s ** 3)))


def _loop(X, W, b, gelu, acc=np.float64, klimit=None, bias_after=False, bias_index="n",
          transpose=False, gelu_fn=_gelu_np):
    X = X.astype(np.float64)
    W = W.astype(np.float64)
    if transpose:
        if W.shape[0] != W.shape[1]:
            raise ValueError("transposed-W mutant needs a square W")
        W = W.T
    M, K = X.shape
    N = W.shape[0]
    Y = np.zeros((M, N))
    kk = K if klimit is None else klimit(K)
    for m in range(M):
        for n in range(N):
            s = acc(0.0)
            for k in range(kk):
                s = acc(s + acc(X[m, k]) * acc(W[n, k]))
            s = float(s)
            bv = 0.0
            if b is not None:
                bv = float(b[n] if bias_index == "n" else b[m % len(b)])
            if not bias_after:
                s += bv
            if gelu:
                s = float(gelu_fn(np.float64(s)))
            if bias_after:
                s += bv
            Y[m, n] = s
    return Y


MUTANTS = {
    "transposed_W": lambda X, W, b, g: _loop(X, W, b, g, transpose=True),
    "drops_last_k": lambda X, W, b, g: _loop(X, W, b, g, klimit=lambda K: max(K - 1, 0)),
    "fp32_accumulator": lambda X, W, b, g: _loop(X, W, b, g, acc=np.float32),
    "bias_after_gelu": lambda X, W, b, g: _loop(X, W, b, g, bias_after=True),
    "bias_indexed_by_row": lambda X, W, b, g: _loop(X, W, b, g, bias_index="m"),
    "no_bias": lambda X, W, b, g: _loop(X, W, None, g),
    "gelu_const_0p0447": lambda X, W, b, g: _loop(X, W, b, g, gelu_fn=lambda s: _gelu_np(s, c3=0.0447)),
    "gelu_sqrt2_over_pi": lambda X, W, b, g: _loop(
        X, W, b, g, gelu_fn=lambda s: _gelu_np(s, c1=math.sqrt(2.0) / math.pi)),
    "gelu_no_half": lambda X, W, b, g: _loop(X, W, b, g, gelu_fn=lambda s: _gelu_np(s, half=1.0)),
}


def test_mutants_reference_is_sound():
    """The loop used by the mutants, unmutated, passes every pin (so a failing
    mutant fails because of its planted mistake)."""
    for pin in LINEAR_PINS:
        pin(lambda X, W, b, g: _loop(X, W, b, g))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mutant = MUTANTS[name]
    caught = []
    for pin in LINEAR_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"


# ------------------------------------------------------------ calibration ---

def test_metric_separates_reorder_from_bug():
    X = si.uniform_pm1(0, 1, (256, 4096))
    W = si.uniform_pm1(0, 2, (256, 4096))
    ref = oracle.linear(X, W)
    y32 = (X @ W.T).astype(np.float64)  # fp32 sums in BLAS order
    e = oracle.rel_err(y32, ref)
    assert 1e-9 < e < 1e-5, e
    bad = ref.copy()
    bad[:64, :64], bad[64:128, 64:128] = ref[64:128, 64:128], ref[:64, :64]
    assert oracle.rel_err(bad, ref) > 5e-2


def test_rel_err_definition():
    assert oracle.rel_err(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == 0.5
    assert oracle.rel_err(np.array([0.5]), np.array([0.0])) == 0.5
    assert oracle.rel_err(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0


# -------------------------------------------------------------- backward ---

from oracle_pins import BACKWARD_PINS, pin_backward_closed_forms, pin_backward_finite_differences, \
    pin_gelu_grad_function  # noqa: E402

REAL_BWD = (lambda X, W, b, dY, g: oracle.backward_dz(X, W, dY, b, g),
            lambda dZ, W: oracle.backward_dx(dZ, W),
            lambda dZ, X: oracle.backward_dw(dZ, X))


def test_gelu_grad_meets_pin():
    pin_gelu_grad_function(oracle.gelu_grad, oracle.gelu)


@pytest.mark.parametrize("pin", BACKWARD_PINS, ids=lambda p: p.__name__)
def test_backward_meets_pin(pin):
    if pin is pin_backward_finite_differences:
        pin(real, REAL_BWD)
    else:
        pin(REAL_BWD)


def test_gelu_backward_matches_dz():
    """The elementwise form (given Z) equals the recomputing form."""
    X = si.normal(9, 1, (6, 40))
    W = si.normal(9, 2, (11, 40), 0.0, 0.2)
    b = si.normal(9, 3, (11,), 0.0, 0.1)
    dY = si.normal(9, 4, (6, 11))
    Z = oracle.linear(X, W, b, False).astype(np.float32)
    ref = oracle.backward_dz(X, W, dY, b, True)
    got = oracle.gelu_backward(dY, Z)
    assert np.max(np.abs(got - ref)) <= 1e-6 * np.max(np.abs(ref))


def _gg_np(z, c3=0.044715, three=3.0, half_sign=1.0):
    c = math.sqrt(2.0 / math.pi)
    t = np.tanh(c * (z + c3 * z ** 3))
    return 0.5 * (1.0 + t) + half_sign * 0.5 * z * (1.0 - t * t) * c * (1.0 + three * c3 * z * z)


def _bwd_np(dz_gelu_grad=_gg_np, dx_transposed=False, dw_transposed=False, db_rows=False, no_grad=False):
    """Numpy restatement with one optional planted mistake."""
    def dz(X, W, b, dY, gelu):
        Z = X.astype(np.float64) @ W.astype(np.float64).T + (0 if b is None else b.astype(np.float64))
        g = dY.astype(np.float64)
        return g * dz_gelu_grad(Z) if (gelu and not no_grad) else g

    def dx(dZ, W):
        dZ, W = dZ.astype(np.float64), W.astype(np.float64)
        if dx_transposed:  # W read as in x out
            return dZ @ W.reshape(W.shape[1], W.shape[0]).T if W.shape[0] != W.shape[1] else dZ @ W.T
        return dZ @ W

    def dw(dZ, X):
        dZ, X = dZ.astype(np.float64), X.astype(np.float64)
        dW = (X.T @ dZ).reshape(dZ.shape[1], X.shape[1]) if dw_transposed else dZ.T @ X
        db = dZ.sum(axis=1)[: dZ.shape[1]] if db_rows else dZ.sum(axis=0)
        if db_rows and db.shape[0] < dZ.shape[1]:
            db = np.resize(db, dZ.shape[1])
        return dW, db
    return dz, dx, dw


BWD_MUTANTS = {
    "dx_transposed_W": _bwd_np(dx_transposed=True),
    "dw_transposed": _bwd_np(dw_transposed=True),
    "db_over_rows": _bwd_np(db_rows=True),
    "gelu_slope_missing": _bwd_np(no_grad=True),
    "gelu_slope_a_not_3a": _bwd_np(dz_gelu_grad=lambda z: _gg_np(z, three=1.0)),
    "gelu_slope_sign": _bwd_np(dz_gelu_grad=lambda z: _gg_np(z, half_sign=-1.0)),
}


def test_backward_mutant_reference_is_sound():
    ref = _bwd_np()
    pin_backward_closed_forms(ref)
    pin_backward_finite_differences(real, ref)


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_pins_catch_mutant(name):
    mutant = BWD_MUTANTS[name]
    caught = False
    for pin in (pin_backward_closed_forms, lambda b: pin_backward_finite_differences(real, b)):
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught = True
    assert caught, f"no backward pin catches mutant {name}"


# ------------------------------------- fused residual, LayerNorm fold, dX through GELU

from oracle_pins import NEXT4_PINS, pin_dx_gelu, pin_fold, pin_layernorm, pin_residual  # noqa: E402

REAL_NEXT4 = {
    pin_residual: (lambda X, W, R, b, g: oracle.linear_residual(X, W, R, b, g),),
    pin_layernorm: (lambda X, g, b, eps: oracle.layernorm(X, g, b, eps),),
    pin_fold: (lambda W, g, bt, b: oracle.fold_layernorm(W, g, bt, b), oracle.layernorm),
    pin_dx_gelu: (lambda dZ, W, Zp: oracle.backward_dx_gelu(dZ, W, Zp),),
}


@pytest.mark.parametrize("pin", NEXT4_PINS, ids=lambda p: p.__name__)
def test_next4_meets_pin(pin):
    pin(*REAL_NEXT4[pin])


def _resid_np(after_act=True, drop=False):
    def fr(X, W, R, b, gelu):
        Z = X.astype(np.float64) @ W.astype(np.float64).T + (0 if b is None else b.astype(np.float64))
        Rd = 0.0 if drop else R.astype(np.float64)
        if not after_act:
            Z = Z + Rd
        Y = _gelu_np(Z) if gelu else Z
        return Y + Rd if after_act else Y
    return fr


def _fold_np(transposed=False, no_bias=False, beta_scaled=False, gamma_on_rows=False):
    def fold(W, gamma, beta=None, bias=None):
        W = W.astype(np.float64)
        g = gamma.astype(np.float64)
        bt = np.zeros(W.shape[1]) if beta is None else beta.astype(np.float64)
        b = np.zeros(W.shape[0]) if (bias is None or no_bias) else bias.astype(np.float64)
        if gamma_on_rows:  # scale row n by gamma[n] (gamma read with the wrong index)
            Wf = W * np.resize(g, W.shape[0])[:, None]
        elif transposed:
            Wf = (W.T * g[:, None]).T.copy() if W.shape[0] == W.shape[1] else W * np.resize(g, W.shape[0])[:, None]
        else:
            Wf = W * g[None, :]
        bf = b + ((W * g[None, :]) @ bt if beta_scaled else W @ bt)
        return Wf, bf
    return fold


def _ln_np(biased=True, eps_outside=False):
    def ln(X, gamma=None, beta=None, eps=1e-5):
        X = X.astype(np.float64)
        mu = X.mean(axis=1, keepdims=True)
        var = X.var(axis=1, keepdims=True, ddof=0 if biased else 1)
        xh = (X - mu) / (np.sqrt(var) + eps if eps_outside else np.sqrt(var + eps))
        if gamma is not None:
            xh = xh * gamma.astype(np.float64)
        if beta is not None:
            xh = xh + beta.astype(np.float64)
        return xh
    return ln


def _dxg_np(no_slope=False, slope_of_dx=False):
    def dxg(dZ, W, Zp):
        dx = dZ.astype(np.float64) @ W.astype(np.float64)
        if no_slope:
            return dx
        return dx * _gg_np(dx if slope_of_dx else Zp.astype(np.float64))
    return dxg


NEXT4_MUTANTS = {
    "residual_before_activation": (pin_residual, (_resid_np(after_act=False),)),
    "residual_dropped": (pin_residual, (_resid_np(drop=True),)),
    "layernorm_unbiased_variance": (pin_layernorm, (_ln_np(biased=False),)),
    "layernorm_eps_outside_root": (pin_layernorm, (_ln_np(eps_outside=True),)),
    "fold_gamma_on_rows": (pin_fold, (_fold_np(gamma_on_rows=True), _ln_np())),
    "fold_bias_dropped": (pin_fold, (_fold_np(no_bias=True), _ln_np())),
    "fold_beta_scaled_by_gamma": (pin_fold, (_fold_np(beta_scaled=True), _ln_np())),
    "dx_gelu_slope_missing": (pin_dx_gelu, (_dxg_np(no_slope=True),)),
    "dx_gelu_slope_of_wrong_tensor": (pin_dx_gelu, (_dxg_np(slope_of_dx=True),)),
}


def test_next4_mutant_references_are_sound():
    pin_residual(_resid_np())
    pin_layernorm(_ln_np())
    pin_fold(_fold_np(), _ln_np())
    pin_dx_gelu(_dxg_np())


@pytest.mark.parametrize("name", sorted(NEXT4_MUTANTS))
def test_next4_pins_catch_mutant(name):
    pin, args = NEXT4_MUTANTS[name]
    with pytest.raises(AssertionError):
        pin(*args)


# ------------------------------------------------------------------ self-attention

from oracle_pins import ATTENTION_PINS  # noqa: E402


def _real_attention(qkv, B, T, H, D, causal, scale):
    return oracle.attention(qkv, B, T, H, D, causal, scale, with_lse=True)


@pytest.mark.parametrize("pin", ATTENTION_PINS, ids=lambda p: p.__name__)
def test_attention_meets_pin(pin):
    pin(_real_attention)


def _attn_np(scale_ignored=False, off_by_one=False, mask_missing=False, v_from_k=False, swap_kv_offsets=False,
             divide_by_max=False, lse_without_max=False):
    def attn(qkv, B, T, H, D, causal, scale):
        C = H * D
        x = qkv.astype(np.float64)
        out = np.zeros((B * T, C))
        lse = np.zeros((B, H, T))
        ko, vo = (2 * C, C) if swap_kv_offsets else (C, 2 * C)
        if v_from_k:
            vo = ko
        sc = 1.0 if scale_ignored else scale
        for b in range(B):
            for h in range(H):
                q = x[b * T:(b + 1) * T, h * D:(h + 1) * D]
                k = x[b * T:(b + 1) * T, ko + h * D:ko + (h + 1) * D]
                v = x[b * T:(b + 1) * T, vo + h * D:vo + (h + 1) * D]
                s = (q @ k.T) * sc
                if causal and not mask_missing:
                    s = np.where(np.tril(np.ones((T, T)), -1 if off_by_one else 0) > 0, s, -np.inf)
                    if off_by_one:
                        s[0, 0] = 0.0  # the first query would see nothing: keep the row finite
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                l = e.sum(axis=1, keepdims=True)
                out[b * T:(b + 1) * T, h * D:(h + 1) * D] = (e @ v) / (np.max(e, axis=1, keepdims=True)
                                                                    if divide_by_max else l)
                lse[b, h] = (np.log(l) if lse_without_max else m + np.log(l))[:, 0]
        return out, lse
    return attn


ATTENTION_MUTANTS = {
    "scale_ignored": _attn_np(scale_ignored=True),
    "causal_mask_off_by_one": _attn_np(off_by_one=True),
    "causal_mask_missing": _attn_np(mask_missing=True),
    "values_read_from_keys": _attn_np(v_from_k=True),
    "k_and_v_offsets_swapped": _attn_np(swap_kv_offsets=True),
    "divided_by_max_not_sum": _attn_np(divide_by_max=True),
    "lse_without_row_max": _attn_np(lse_without_max=True),
}


def test_attention_mutant_reference_is_sound():
    ref = _attn_np()
    for pin in ATTENTION_PINS:
        pin(ref)


@pytest.mark.parametrize("name", sorted(ATTENTION_MUTANTS))
def test_attention_pins_catch_mutant(name):
    mutant = ATTENTION_MUTANTS[name]
    caught = False
    for pin in ATTENTION_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
    assert caught, f"no attention pin catches mutant {name}"
