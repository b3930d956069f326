"""GB300 linear layer: Y = act(X . W^T + bias), W stored out x in.

A thin ctypes binding over the C ABI in ``include/lin.h`` (library
``_build/liblin.so``, built by :func:`build`). The binding only marshals
arguments: torch supplies device memory and the current CUDA stream, and every
step of the multiply runs in this package's CUDA kernels. There is no CPU path:
if the library is missing or the GPU call fails, an exception is raised.

    import torch, transformer_linear_layer_gb300 as tll
    y = tll.forward(x_bf16, w_bf16, bias_fp32, epilogue="gelu")   # -> bf16
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB as _LIB_PATH
from .build import TIMELINE_LIB as _TIMELINE_LIB_PATH
from .build import build

__all__ = [
    "LinError", "Context", "Plan", "forward", "forward_plan", "plan_query", "plan_make", "build",
    "backward_data", "backward_weight", "gelu_backward", "attention_forward",
    "library", "PREC_FP32", "PREC_TF32", "PREC_BF16", "EPI_NONE", "EPI_GELU_TANH",
    "KERNEL_NONE", "KERNEL_FILL", "KERNEL_SKINNY", "KERNEL_FFMA", "KERNEL_TC", "KERNEL_GEMV",
]

PREC_FP32, PREC_TF32, PREC_BF16 = 0, 1, 2
EPI_NONE, EPI_GELU_TANH = 0, 1
KERNEL_NONE, KERNEL_FILL, KERNEL_SKINNY, KERNEL_FFMA, KERNEL_TC, KERNEL_GEMV = 0, 1, 2, 3, 4, 5
KERNEL_NAMES = {0: "none", 1: "fill", 2: "skinny", 3: "ffma", 4: "tc", 5: "gemv"}
OPT_EARLY_START = 1
OPT_ADAPTIVE_PLANS = 2
OPT_PROGRAMMATIC_LAUNCH = 3
# LIN_OPT_EARLY_START levels: nothing before the previous kernel finishes (the
# default); W and bias may be read early; X too (only when no other work on the
# stream writes a call's inputs between library calls).
EARLY_NONE, EARLY_WEIGHTS, EARLY_ALL = 0, 1, 2
OK, ERR_ARG, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
# LIN_STATIC_SCRATCH_BYTES: the fixed device array behind lin_forward_fp32_static.
STATIC_SCRATCH_BYTES = 8 << 20

_PREC_NAMES = {"fp32": PREC_FP32, "tf32": PREC_TF32, "bf16": PREC_BF16}
_EPI_NAMES = {"none": EPI_NONE, None: EPI_NONE, "gelu": EPI_GELU_TANH, "gelu_tanh": EPI_GELU_TANH}


class Plan(ctypes.Structure):
    """Mirror of ``lin_plan``."""

    _fields_ = [
        ("kernel", ctypes.c_int), ("variant", ctypes.c_int), ("bm", ctypes.c_int), ("bn", ctypes.c_int),
        ("bk", ctypes.c_int), ("splits", ctypes.c_int), ("stages", ctypes.c_int), ("grid_x", ctypes.c_int),
        ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int), ("threads", ctypes.c_int),
        ("workspace_bytes", ctypes.c_longlong),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        return d

    def __repr__(self):
        return f"Plan({self.as_dict()})"


class LinError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = library().lin_strerror(status).decode()
        super().__init__(f"{what}: status {status} ({msg})" if what else f"status {status} ({msg})")


_lock = threading.Lock()
_lib = None


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built ({_LIB_PATH} missing); run "
                    "`python -m transformer_linear_layer_gb300.build` or __graft_entry__.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            PP = ctypes.POINTER(Plan)
            sig = {
                "lin_create": ([ctypes.POINTER(P), I, Z], I),
                "lin_destroy": ([P], I),
                "lin_forward": ([P, I, I, I, P, P, P, P, I, I, P], I),
                "lin_forward_plan": ([P, PP, I, I, I, P, P, P, P, I, I, P], I),
                "lin_plan_query": ([I, I, I, I, I, I, Z, PP], I),
                "lin_plan_make": ([I, I, I, I, I, I, I, I, PP], I),
                "lin_check_device": ([P, P], I),
                "lin_ctx_info": ([P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(Z)], I),
                "lin_set_option": ([P, I, ctypes.c_longlong], I),
                "lin_ctx_last_plan": ([P, PP], I),
                "lin_forward_fp32_static": ([I, I, I, P, P, P, P, I, P], I),
                "lin_backward_data": ([P, I, I, I, P, P, P, I, P], I),
                "lin_backward_weight": ([P, I, I, I, P, P, P, P, I, P], I),
                "lin_gelu_backward": ([P, ctypes.c_longlong, P, P, P, I, P], I),
                "lin_forward_residual": ([P, I, I, I, P, P, P, P, P, I, I, P], I),
                "lin_plan_check": ([PP, I, I, I, I, ctypes.c_size_t], I),
                "lin_backward_data_gelu": ([P, I, I, I, P, P, P, P, I, P], I),
                "lin_fold_layernorm": ([P, I, I, P, P, P, P, P, P, I, P], I),
                "lin_set_plan_override": ([P, I, I, I, I, I, PP], I),
                "lin_clear_plan_overrides": ([P], I),
                "lin_probe_ffma": ([P, I, P, ctypes.POINTER(ctypes.c_double), P], I),
                "lin_timeline": ([I, P, Z, I], I),
                "lin_attention_forward": ([P, I, I, I, I, P, P, P, I, ctypes.c_float, P], I),
                "lin_strerror": ([I], ctypes.c_char_p),
                "lin_abi_version": ([], I),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


# Shape of a kernel timeline array (LIN_TIMELINE_CTAS x LIN_TIMELINE_SLOTS),
# and the timeline id of the attention kernel (LIN_TIMELINE_ATTENTION).
TIMELINE_CTAS, TIMELINE_SLOTS = 1024, 192
TIMELINE_ATTENTION = 16


def use_timeline_build() -> str:
    """Build (if stale) the timeline library (kernels compiled with
    -DLIN_TIMELINE) and load it instead of the library build. Call before the
    first library call of the process; returns the library path."""
    global _LIB_PATH
    path = build(timeline=True)
    with _lock:
        if _lib is not None and _LIB_PATH != path:
            raise RuntimeError("the library build is already loaded in this process")
        _LIB_PATH = path
    return path


def timeline(kernel: int, clear: bool = True):
    """The stamp array of ``kernel`` (KERNEL_TC, KERNEL_SKINNY or
    TIMELINE_ATTENTION) as an int64
    numpy array of TIMELINE_CTAS x TIMELINE_SLOTS nanoseconds (0 = not
    reached), synchronously; zeroes it afterwards if ``clear``. Needs the
    timeline build (:func:`use_timeline_build`)."""
    import numpy as np

    buf = np.zeros(TIMELINE_CTAS * TIMELINE_SLOTS, dtype=np.uint64)
    rc = library().lin_timeline(kernel, buf.ctypes.data, buf.nbytes, 1 if clear else 0)
    if rc != OK:
        raise LinError(rc, "lin_timeline")
    return buf.reshape(TIMELINE_CTAS, TIMELINE_SLOTS).astype(np.int64)


def timeline_clear(kernel: int):
    """Zero a kernel's stamp array (timeline build only)."""
    rc = library().lin_timeline(kernel, None, 0, 1)
    if rc != OK:
        raise LinError(rc, "lin_timeline")


def _prec(p) -> int:
    return _PREC_NAMES[p] if isinstance(p, str) else int(p)


def _epi(e) -> int:
    return _EPI_NAMES[e] if (e is None or isinstance(e, str)) else int(e)


def plan_query(sm_count: int, M: int, N: int, K: int, precision="bf16", epilogue="none",
               workspace_bytes: int = 64 << 20) -> Plan:
    """The dispatch table's plan for a shape (host only, no GPU needed)."""
    p = Plan()
    rc = library().lin_plan_query(sm_count, M, N, K, _prec(precision), _epi(epilogue), workspace_bytes,
                                  ctypes.byref(p))
    if rc != OK:
        raise LinError(rc, "lin_plan_query")
    return p


def plan_make(sm_count: int, kernel: int, variant: int, splits: int, M: int, N: int, K: int,
              precision="bf16") -> Plan:
    """A plan for one kernel family / tile configuration (host only)."""
    p = Plan()
    rc = library().lin_plan_make(sm_count, kernel, variant, splits, M, N, K, _prec(precision), ctypes.byref(p))
    if rc != OK:
        raise LinError(rc, "lin_plan_make")
    return p


def plan_check(plan: Plan, M: int, N: int, K: int, precision="bf16", workspace_bytes: int = 64 << 20) -> int:
    """Status lin_forward_plan would return for this plan and shape (host only;
    0 = accepted)."""
    return library().lin_plan_check(ctypes.byref(plan), M, N, K, _prec(precision), workspace_bytes)


class Context:
    """Owns a ``lin_ctx``: device, split-K workspace and the device status word."""

    def __init__(self, device: int = 0, workspace_bytes: int = 0):
        self._h = ctypes.c_void_p()
        rc = library().lin_create(ctypes.byref(self._h), int(device), int(workspace_bytes))
        if rc != OK:
            raise LinError(rc, "lin_create")
        dev, sms, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
        library().lin_ctx_info(self._h, ctypes.byref(dev), ctypes.byref(sms), ctypes.byref(ws))
        self.device, self.sm_count, self.workspace_bytes = dev.value, sms.value, ws.value

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            library().lin_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def check(self, stream=None):
        """Synchronise and raise if a kernel reported a timeout (status word)."""
        rc = library().lin_check_device(self._h, _stream_ptr(stream, self.device))
        if rc != OK:
            raise LinError(rc, "lin_check_device")

    def set_option(self, option: int, value: int):
        rc = library().lin_set_option(self._h, int(option), int(value))
        if rc != OK:
            raise LinError(rc, "lin_set_option")

    def last_plan(self) -> Plan:
        """The plan of the last call launched through this context."""
        p = Plan()
        rc = library().lin_ctx_last_plan(self._h, ctypes.byref(p))
        if rc != OK:
            raise LinError(rc, "lin_ctx_last_plan")
        return p

    def plan(self, M, N, K, precision="bf16", epilogue="none") -> Plan:
        """The built-in table's plan (installed overrides are not consulted)."""
        return plan_query(self.sm_count, M, N, K, precision, epilogue, self.workspace_bytes)

    def set_override(self, M, N, K, precision, epilogue, plan: Plan | None):
        """Install (or, with None, remove) the plan lin_forward uses for this call signature."""
        rc = library().lin_set_plan_override(self._h, M, N, K, _prec(precision), _epi(epilogue),
                                             None if plan is None else ctypes.byref(plan))
        if rc != OK:
            raise LinError(rc, "lin_set_plan_override")

    def clear_overrides(self):
        rc = library().lin_clear_plan_overrides(self._h)
        if rc != OK:
            raise LinError(rc, "lin_clear_plan_overrides")

    # raw-pointer calls (the C ABI, one to one) ---------------------------------
    def forward_ptr(self, M, N, K, X, W, bias, Y, epilogue, precision, stream) -> int:
        return library().lin_forward(self._h, M, N, K, X, W, bias, Y, _epi(epilogue), _prec(precision), stream)

    def probe_ffma_ptr(self, iters: int, out, stream) -> float:
        """Launch the fp32 FMA throughput probe (lin_probe_ffma) on `stream`;
        returns the FLOPs launched. The caller times it."""
        flops = ctypes.c_double()
        rc = library().lin_probe_ffma(self._h, int(iters), out, ctypes.byref(flops), stream)
        if rc != OK:
            raise LinError(rc, "lin_probe_ffma")
        return flops.value

    def forward_plan_ptr(self, plan: Plan, M, N, K, X, W, bias, Y, epilogue, precision, stream) -> int:
        return library().lin_forward_plan(self._h, ctypes.byref(plan), M, N, K, X, W, bias, Y, _epi(epilogue),
                                          _prec(precision), stream)


def _stream_ptr(stream, device):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_contexts: dict = {}


def default_context(device: int) -> Context:
    with _lock:
        ctx = _contexts.get(device)
    if ctx is None:
        ctx = Context(device)
        with _lock:
            _contexts.setdefault(device, ctx)
            ctx = _contexts[device]
    return ctx


def _marshal(x, w, bias, out, precision):
    import torch

    prec = precision
    if prec is None:
        prec = "bf16" if x.dtype == torch.bfloat16 else "fp32"
    prec = _prec(prec)
    want = torch.bfloat16 if prec == PREC_BF16 else torch.float32
    if x.dtype != want or w.dtype != want:
        raise TypeError(f"precision {prec} needs {want} X and W, got {x.dtype} and {w.dtype}")
    if not (x.is_cuda and w.is_cuda):
        raise ValueError("X and W must be CUDA tensors")
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"need X (M x K) and W (N x K), got {tuple(x.shape)} and {tuple(w.shape)}")
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("X and W must be contiguous row-major")
    M, K = x.shape
    N = w.shape[0]
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.shape != (N,) or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32 CUDA vector of length N")
    if out is None:
        out = torch.empty((M, N), dtype=want, device=x.device)
    elif out.dtype != want or out.shape != (M, N) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous M x N CUDA tensor of the output dtype")
    return prec, M, N, K, out


def forward(x, w, bias=None, epilogue="none", precision=None, out=None, ctx: Context | None = None, stream=None):
    """Y = act(x . w^T + bias) on x's device, asynchronously on the current stream.

    x: M x K, w: N x K (bf16 for precision "bf16", fp32 for "fp32"/"tf32"),
    bias: fp32 length N or None, epilogue: "none" | "gelu". Returns Y (M x N).
    """
    prec, M, N, K, out = _marshal(x, w, bias, out, precision)
    dev = x.device.index if x.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = ctx.forward_ptr(M, N, K, x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                         out.data_ptr(), epilogue, prec, _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_forward")
    return out


def forward_residual(x, w, residual, bias=None, epilogue="none", precision=None, out=None,
                     ctx: Context | None = None, stream=None):
    """Y = act(x . w^T + bias) + residual, the add in the GEMM's store.
    ``out`` may be ``residual`` itself (x = x + layer(h) in place); by
    default Y is a new tensor."""
    prec, M, N, K, out = _marshal(x, w, bias, out, precision)
    _check(residual, out.dtype, (M, N), "residual")
    dev = x.device.index if x.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_forward_residual(ctx._h, M, N, K, x.data_ptr(), w.data_ptr(),
                                        None if bias is None else bias.data_ptr(), residual.data_ptr(),
                                        out.data_ptr(), _epi(epilogue), prec, _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_forward_residual")
    return out


def fold_layernorm(w, gamma, beta=None, bias=None, precision="fp32", w_out=None, bias_out=None,
                   ctx: Context | None = None, stream=None):
    """The next layer's (W, bias) with a LayerNorm's scale and shift folded in,
    computed on the device in double: W_out = w diag(gamma), bias_out =
    bias + w beta. ``w`` (N x K), ``gamma``, ``beta`` and ``bias`` are fp32;
    W_out has the storage type of ``precision``. Returns (W_out, bias_out)."""
    import torch

    N, K = w.shape
    _check(w, torch.float32, (N, K), "w")
    _check(gamma, torch.float32, (K,), "gamma")
    if beta is not None:
        _check(beta, torch.float32, (K,), "beta")
    if bias is not None:
        _check(bias, torch.float32, (N,), "bias")
    prec = _prec(precision)
    wdt = torch.bfloat16 if prec == PREC_BF16 else torch.float32
    if w_out is None:
        w_out = torch.empty((N, K), dtype=wdt, device=w.device)
    _check(w_out, wdt, (N, K), "w_out")
    if bias_out is None:
        bias_out = torch.empty((N,), dtype=torch.float32, device=w.device)
    _check(bias_out, torch.float32, (N,), "bias_out")
    dev = w.device.index if w.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_fold_layernorm(ctx._h, N, K, w.data_ptr(), None if bias is None else bias.data_ptr(),
                                      gamma.data_ptr(), None if beta is None else beta.data_ptr(), w_out.data_ptr(),
                                      bias_out.data_ptr(), prec, _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_fold_layernorm")
    return w_out, bias_out


def forward_plan(plan: Plan, x, w, bias=None, epilogue="none", precision=None, out=None,
                 ctx: Context | None = None, stream=None):
    """As :func:`forward` with an explicit launch configuration."""
    prec, M, N, K, out = _marshal(x, w, bias, out, precision)
    dev = x.device.index if x.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = ctx.forward_plan_ptr(plan, M, N, K, x.data_ptr(), w.data_ptr(),
                              None if bias is None else bias.data_ptr(), out.data_ptr(), epilogue, prec,
                              _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_forward_plan")
    return out


# ---------------------------------------------------------------- backward

def _bwd_dtype(t, precision):
    import torch

    prec = precision
    if prec is None:
        prec = "bf16" if t.dtype == torch.bfloat16 else "fp32"
    prec = _prec(prec)
    return prec, (torch.bfloat16 if prec == PREC_BF16 else torch.float32)


def _check(t, want, shape, what):
    if t.dtype != want or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must be a contiguous {want} CUDA tensor of shape {tuple(shape)}")


def backward_data(dz, w, out=None, precision=None, ctx: Context | None = None, stream=None):
    """dX (M x K) = dz (M x N) . w (N x K): the input gradient of the layer
    (dz = dY times the activation's slope)."""
    import torch

    prec, want = _bwd_dtype(dz, precision)
    M, N = dz.shape
    K = w.shape[1]
    _check(dz, want, (M, N), "dz")
    _check(w, want, (N, K), "w")
    if out is None:
        out = torch.empty((M, K), dtype=want, device=dz.device)
    _check(out, want, (M, K), "out")
    dev = dz.device.index if dz.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_backward_data(ctx._h, M, N, K, dz.data_ptr(), w.data_ptr(), out.data_ptr(), prec,
                                     _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_backward_data")
    return out


def backward_data_gelu(dz, w, zp, out=None, precision=None, ctx: Context | None = None, stream=None):
    """dZp (M x K) = (dz . w) * gelu'(zp): the input gradient carried through
    the GELU that made this layer's input from the previous layer's
    pre-activation ``zp`` (M x K), in one pass. ``out`` may be ``zp``."""
    import torch

    prec, want = _bwd_dtype(dz, precision)
    M, N = dz.shape
    K = w.shape[1]
    _check(dz, want, (M, N), "dz")
    _check(w, want, (N, K), "w")
    _check(zp, want, (M, K), "zp")
    if out is None:
        out = torch.empty((M, K), dtype=want, device=dz.device)
    _check(out, want, (M, K), "out")
    dev = dz.device.index if dz.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_backward_data_gelu(ctx._h, M, N, K, dz.data_ptr(), w.data_ptr(), zp.data_ptr(),
                                          out.data_ptr(), prec, _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_backward_data_gelu")
    return out


def backward_weight(dz, x, out=None, db=None, precision=None, ctx: Context | None = None, stream=None):
    """dW (N x K) = dz^T . x (dz: M x N, x: M x K) and, when ``db`` is True or
    an fp32 tensor of length N, db = the column sums of dz. Returns (dW, db)."""
    import torch

    prec, want = _bwd_dtype(dz, precision)
    M, N = dz.shape
    K = x.shape[1]
    _check(dz, want, (M, N), "dz")
    _check(x, want, (M, K), "x")
    if out is None:
        out = torch.empty((N, K), dtype=want, device=dz.device)
    _check(out, want, (N, K), "out")
    if db is True:
        db = torch.empty((N,), dtype=torch.float32, device=dz.device)
    if db is not None and db is not False:
        _check(db, torch.float32, (N,), "db")
    else:
        db = None
    dev = dz.device.index if dz.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_backward_weight(ctx._h, M, N, K, dz.data_ptr(), x.data_ptr(), out.data_ptr(),
                                       None if db is None else db.data_ptr(), prec, _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_backward_weight")
    return out, db


def gelu_backward(dy, z, out=None, precision=None, ctx: Context | None = None, stream=None):
    """dZ = dy * gelu'(z) (z: the forward's pre-activation), elementwise."""
    import torch

    prec, want = _bwd_dtype(dy, precision)
    _check(dy, want, tuple(dy.shape), "dy")
    _check(z, want, tuple(dy.shape), "z")
    if out is None:
        out = torch.empty_like(dy)
    _check(out, want, tuple(dy.shape), "out")
    dev = dy.device.index if dy.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_gelu_backward(ctx._h, dy.numel(), dy.data_ptr(), z.data_ptr(), out.data_ptr(), prec,
                                     _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_gelu_backward")
    return out


# ---------------------------------------------------------------- attention

def attention_forward(qkv, B: int, T: int, H: int, causal: bool = True, scale: float | None = None, out=None,
                      lse=None, with_lse: bool = False, ctx: Context | None = None, stream=None):
    """Fused self-attention forward from the qkv projection's output.

    qkv: contiguous bf16 CUDA tensor of (B*T) x 3C (C = 64 H; q, k, v at
    column offsets 0, C, 2C, head h at 64 h within each). Returns out
    ((B*T) x C bf16), or (out, lse) with lse (B, H, T) fp32 when ``with_lse``
    or an lse tensor is given. scale defaults to 1/sqrt(64)."""
    import torch

    D = 64
    C = H * D
    _check(qkv, torch.bfloat16, (B * T, 3 * C), "qkv")
    if out is None:
        out = torch.empty((B * T, C), dtype=torch.bfloat16, device=qkv.device)
    _check(out, torch.bfloat16, (B * T, C), "out")
    if lse is None and with_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=qkv.device)
    if lse is not None:
        _check(lse, torch.float32, (B, H, T), "lse")
    dev = qkv.device.index if qkv.device.index is not None else 0
    ctx = ctx or default_context(dev)
    rc = library().lin_attention_forward(ctx._h, B, T, H, D, qkv.data_ptr(), out.data_ptr(),
                                         None if lse is None else lse.data_ptr(), int(bool(causal)),
                                         0.0 if scale is None else float(scale), _stream_ptr(stream, dev))
    if rc != OK:
        raise LinError(rc, "lin_attention_forward")
    return (out, lse) if lse is not None else out
