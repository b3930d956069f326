"""CPU oracle for Y = act(X . W^T + bias), its backward, the fused residual,
the LayerNorm fold, the dX carried through a GELU and the self-attention that
reads the qkv projection. TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package. The library under ``transformer_linear_layer_gb300``
never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation in
ascending k); this module compiles it with gcc on first use and wraps it with
ctypes. :func:`rel_err` is the acceptance metric the pages use for a matmul:
the worst absolute error over max|Y_ref| ("Writing a CUDA matmul that catches
cuBLAS", section "The measurement was nearly wrong").

Every oracle function here is pinned by ``tests/test_oracle_pins.py`` against
identity and permutation weights, exact small-integer products, brute force on
tiny shapes and an independent library GELU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

TOL = {0: 1e-5, 1: 5e-3, 2: 1e-2}  # fp32, tf32, bf16 inputs (acceptance bars)


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP if present)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", _SRC, "-lm"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_linear.argtypes = [i64, i64, i64, p, p, p, ctypes.c_int, p, ctypes.c_int]
            lib.oracle_linear.restype = None
            lib.oracle_linear_entries.argtypes = [i64, p, p, i64, p, p, p, ctypes.c_int, p, ctypes.c_int]
            lib.oracle_linear_entries.restype = None
            lib.oracle_gelu_array.argtypes = [i64, p, p]
            lib.oracle_gelu_array.restype = None
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_backward_dz.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int, p, ctypes.c_int]
            lib.oracle_backward_dz.restype = None
            lib.oracle_gelu_backward.argtypes = [i64, p, p, p]
            lib.oracle_gelu_backward.restype = None
            lib.oracle_backward_dx.argtypes = [i64, i64, i64, p, p, p, ctypes.c_int]
            lib.oracle_backward_dx.restype = None
            lib.oracle_backward_dw.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_backward_dw.restype = None
            lib.oracle_gelu_grad_array.argtypes = [i64, p, p]
            lib.oracle_gelu_grad_array.restype = None
            lib.oracle_linear_residual.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int, p, ctypes.c_int]
            lib.oracle_linear_residual.restype = None
            lib.oracle_layernorm.argtypes = [i64, i64, p, p, p, ctypes.c_double, p]
            lib.oracle_layernorm.restype = None
            lib.oracle_fold_layernorm.argtypes = [i64, i64, p, p, p, p, p, p]
            lib.oracle_fold_layernorm.restype = None
            lib.oracle_backward_dx_gelu.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_backward_dx_gelu.restype = None
            lib.oracle_attention.argtypes = [i64, i64, i64, i64, p, ctypes.c_int, ctypes.c_double, p, p, ctypes.c_int]
            lib.oracle_attention.restype = None
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def linear(X, W, bias=None, gelu: bool = False, nthreads: int = 0) -> np.ndarray:
    """Y (float64, M x N) = act(X . W^T + bias); X: M x K, W: N x K (fp32 values)."""
    X, W = _f32(X), _f32(W)
    M, K = X.shape
    N, K2 = W.shape
    assert K == K2, "X and W disagree on K"
    b = None if bias is None else _f32(bias)
    if b is not None:
        assert b.shape == (N,)
    Y = np.empty((M, N), dtype=np.float64)
    _load().oracle_linear(M, N, K, X.ctypes.data, W.ctypes.data,
                          None if b is None else b.ctypes.data, int(bool(gelu)), Y.ctypes.data, int(nthreads))
    return Y


def linear_entries(X, W, ms, ns, bias=None, gelu: bool = False, nthreads: int = 0) -> np.ndarray:
    """Selected outputs Y[ms[i], ns[i]] (float64), computed one by one."""
    X, W = _f32(X), _f32(W)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms.shape == ns.shape
    assert X.shape[1] == W.shape[1]
    assert ms.size == 0 or (ms.min() >= 0 and ms.max() < X.shape[0] and ns.min() >= 0 and ns.max() < W.shape[0])
    b = None if bias is None else _f32(bias)
    out = np.empty(ms.shape, dtype=np.float64)
    _load().oracle_linear_entries(ms.size, ms.ctypes.data, ns.ctypes.data, X.shape[1], X.ctypes.data,
                                  W.ctypes.data, None if b is None else b.ctypes.data, int(bool(gelu)),
                                  out.ctypes.data, int(nthreads))
    return out


def gelu(x) -> np.ndarray:
    """The oracle's tanh-form GELU on a float64 array."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().oracle_gelu_array(x.size, x.ctypes.data, out.ctypes.data)
    return out


def backward_dz(X, W, dY, bias=None, gelu: bool = False, nthreads: int = 0) -> np.ndarray:
    """dZ (float64, M x N) = dY * act'(X . W^T + bias)."""
    X, W, dY = _f32(X), _f32(W), _f32(dY)
    M, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K and dY.shape == (M, N)
    b = None if bias is None else _f32(bias)
    out = np.empty((M, N), dtype=np.float64)
    _load().oracle_backward_dz(M, N, K, X.ctypes.data, W.ctypes.data, None if b is None else b.ctypes.data,
                               dY.ctypes.data, int(bool(gelu)), out.ctypes.data, int(nthreads))
    return out


def gelu_backward(dY, Z) -> np.ndarray:
    """dZ (float64) = dY * gelu'(Z), elementwise; dY and Z hold fp32 values."""
    dY, Z = _f32(dY), _f32(Z)
    assert dY.shape == Z.shape
    out = np.empty(dY.shape, dtype=np.float64)
    _load().oracle_gelu_backward(dY.size, dY.ctypes.data, Z.ctypes.data, out.ctypes.data)
    return out


def backward_dx(dZ, W, nthreads: int = 0) -> np.ndarray:
    """dX (float64, M x K) = dZ . W; dZ: M x N, W: N x K (fp32 values)."""
    dZ, W = _f32(dZ), _f32(W)
    M, N = dZ.shape
    N2, K = W.shape
    assert N == N2
    out = np.empty((M, K), dtype=np.float64)
    _load().oracle_backward_dx(M, N, K, dZ.ctypes.data, W.ctypes.data, out.ctypes.data, int(nthreads))
    return out


def backward_dw(dZ, X, with_bias: bool = True, nthreads: int = 0):
    """(dW (float64, N x K) = dZ^T . X, db (float64, N) = column sums of dZ or
    None); dZ: M x N, X: M x K (fp32 values)."""
    dZ, X = _f32(dZ), _f32(X)
    M, N = dZ.shape
    M2, K = X.shape
    assert M == M2
    dW = np.empty((N, K), dtype=np.float64)
    db = np.empty((N,), dtype=np.float64) if with_bias else None
    _load().oracle_backward_dw(M, N, K, dZ.ctypes.data, X.ctypes.data, dW.ctypes.data,
                               None if db is None else db.ctypes.data, int(nthreads))
    return dW, db


def gelu_grad(x) -> np.ndarray:
    """The oracle's slope of the tanh-form GELU on a float64 array."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().oracle_gelu_grad_array(x.size, x.ctypes.data, out.ctypes.data)
    return out


def linear_residual(X, W, R, bias=None, gelu: bool = False, nthreads: int = 0) -> np.ndarray:
    """Y (float64, M x N) = act(X . W^T + bias) + R; R: M x N (fp32 values)."""
    X, W, R = _f32(X), _f32(W), _f32(R)
    M, K = X.shape
    N, K2 = W.shape
    assert K == K2 and R.shape == (M, N)
    b = None if bias is None else _f32(bias)
    Y = np.empty((M, N), dtype=np.float64)
    _load().oracle_linear_residual(M, N, K, X.ctypes.data, W.ctypes.data, None if b is None else b.ctypes.data,
                                   R.ctypes.data, int(bool(gelu)), Y.ctypes.data, int(nthreads))
    return Y


def layernorm(X, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm over the last axis in float64 (gamma / beta None: xhat alone)."""
    X = _f32(X)
    M, K = X.shape
    g = None if gamma is None else _f32(gamma)
    bt = None if beta is None else _f32(beta)
    out = np.empty((M, K), dtype=np.float64)
    _load().oracle_layernorm(M, K, X.ctypes.data, None if g is None else g.ctypes.data,
                             None if bt is None else bt.ctypes.data, float(eps), out.ctypes.data)
    return out


def fold_layernorm(W, gamma, beta=None, bias=None):
    """(Wf, bf) in float64: the next layer's weight and bias with LayerNorm's
    scale and shift folded in (Wf = W diag(gamma), bf = bias + W beta)."""
    W, g = _f32(W), _f32(gamma)
    N, K = W.shape
    assert g.shape == (K,)
    bt = None if beta is None else _f32(beta)
    b = None if bias is None else _f32(bias)
    Wf = np.empty((N, K), dtype=np.float64)
    bf = np.empty((N,), dtype=np.float64)
    _load().oracle_fold_layernorm(N, K, W.ctypes.data, None if b is None else b.ctypes.data, g.ctypes.data,
                                  None if bt is None else bt.ctypes.data, Wf.ctypes.data, bf.ctypes.data)
    return Wf, bf


def backward_dx_gelu(dZ, W, Zp, nthreads: int = 0) -> np.ndarray:
    """dZp (float64, M x K) = (dZ . W) * gelu'(Zp): dX carried through the GELU
    that produced X from the previous layer's pre-activation Zp (M x K)."""
    dZ, W, Zp = _f32(dZ), _f32(W), _f32(Zp)
    M, N = dZ.shape
    N2, K = W.shape
    assert N == N2 and Zp.shape == (M, K)
    out = np.empty((M, K), dtype=np.float64)
    _load().oracle_backward_dx_gelu(M, N, K, dZ.ctypes.data, W.ctypes.data, Zp.ctypes.data, out.ctypes.data,
                                    int(nthreads))
    return out


def attention(qkv, B: int, T: int, H: int, D: int, causal: bool = True, scale: float | None = None,
              with_lse: bool = False, nthreads: int = 0):
    """Self-attention from the qkv projection's output (float64).

    qkv: (B*T) x 3C fp32 values (C = H*D; q, k, v at column offsets 0, C, 2C,
    head h at h*D within each); returns out ((B*T) x C), and lse (B x H x T,
    the log of each query's softmax denominator plus its row max) when
    ``with_lse``. scale defaults to 1/sqrt(D)."""
    qkv = _f32(qkv)
    assert qkv.shape == (B * T, 3 * H * D)
    sc = 1.0 / float(np.sqrt(D)) if scale is None else float(scale)
    out = np.empty((B * T, H * D), dtype=np.float64)
    lse = np.empty((B, H, T), dtype=np.float64) if with_lse else None
    _load().oracle_attention(B, T, H, D, qkv.ctypes.data, int(bool(causal)), sc, out.ctypes.data,
                             None if lse is None else lse.ctypes.data, int(nthreads))
    return (out, lse) if with_lse else out


def rel_err(y, y_ref) -> float:
    """max|y - y_ref| / max|y_ref| (max|y - y_ref| when y_ref is all zero)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if y.size == 0:
        return 0.0
    num = float(np.max(np.abs(y - y_ref)))
    den = float(np.max(np.abs(y_ref)))
    return num / den if den > 0 else num
