"""The fp32 entry point that allocates nothing (lin_forward_fp32_static).

It serves callers that cannot allocate device memory when they run the layer:
runtimes that reserved all device memory for their own pool, latency-critical
paths where an allocation could block or fail, plug-ins handed device pointers
but no allocator. Its split-K scratch is a fixed array inside the library.

These tests call it through the C ABI, twice in a row (consecutive calls share
that array and it keeps the last call's contents), and check each result
against the CPU oracle at the fp32 tolerance and bit for bit against
lin_forward, which runs the same kernel with the same split from a context's
workspace. The file is named to be collected last, so that a run stopping at
the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll

pytestmark = pytest.mark.gpu

SHAPES = list(si.GPT2_M128_FP32) + [
    si.Layer("ragged", 70, 333, 132, si.PREC_FP32, si.EPI_GELU, bias=True),
    si.SQUARE_256_FP32,
    si.Layer("gemv_rows", 5, 700, 256, si.PREC_FP32, bias=True),
]


def _static(lib, x, w, bias, y, epi):
    return lib.lin_forward_fp32_static(x.shape[0], w.shape[0], x.shape[1], x.data_ptr(), w.data_ptr(),
                                       None if bias is None else bias.data_ptr(), y.data_ptr(), epi,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("layer", SHAPES, ids=lambda l: l.name)
def test_static_scratch_matches_oracle_and_lin_forward(layer):
    lib = tll.library()
    X, W, b = si.make_inputs(layer)
    x = torch.from_numpy(X).cuda()
    w = torch.from_numpy(W).cuda()
    bias = None if b is None else torch.from_numpy(b).cuda()
    epi = tll.EPI_GELU_TANH if layer.epilogue else tll.EPI_NONE
    ref = oracle.linear(X, W, b, bool(layer.epilogue))
    y_ctx = tll.forward(x, w, bias, epilogue=epi, precision="fp32")
    y1 = torch.full((layer.M, layer.N), float("nan"), device="cuda")
    y2 = torch.full((layer.M, layer.N), float("nan"), device="cuda")
    assert _static(lib, x, w, bias, y1, epi) == tll.OK
    assert _static(lib, x, w, bias, y2, epi) == tll.OK  # the second call finds the array as the first left it
    torch.cuda.synchronize()
    for y in (y1, y2):
        got = y.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert oracle.rel_err(got, ref) <= oracle.TOL[si.PREC_FP32]
    # Same kernel, same split, same fixed summation order: the same bits.
    assert torch.equal(y1, y2)
    assert torch.equal(y1, y_ctx)


def test_static_scratch_allocates_nothing():
    """After a first call on the device (which may load the library's module),
    further calls leave the device's free memory unchanged."""
    lib = tll.library()
    layer = si.GPT2_M128_FP32[3]  # fc2: the longest K, a split of the scratch
    X, W, b = si.make_inputs(layer)
    x, w, bias = torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda()
    y = torch.empty((layer.M, layer.N), device="cuda")
    assert _static(lib, x, w, bias, y, tll.EPI_NONE) == tll.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _static(lib, x, w, bias, y, tll.EPI_NONE) == tll.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert oracle.rel_err(y.double().cpu().numpy(), oracle.linear(X, W, b)) <= oracle.TOL[si.PREC_FP32]


def test_gpt2_shapes_exercise_the_split():
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    for layer in si.GPT2_M128_FP32:
        p = tll.plan_query(sm, layer.M, layer.N, layer.K, "fp32", workspace_bytes=1 << 62)
        assert p.splits > 1 and 0 < p.workspace_bytes <= tll.STATIC_SCRATCH_BYTES


def test_static_scratch_refuses_oversized_split():
    """On a device whose dispatch table splits this shape beyond the array
    (the split fills two 64x64 CTAs per SM, so its scratch grows with the SM
    count: ~5 MB at 152 SMs), nothing is launched and LIN_ERR_WORKSPACE comes
    back. The host-side rule is checked without a GPU in test_abi_cpu.py."""
    lib = tll.library()
    M, N, K = 64, 512, 8192
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    need = tll.plan_query(sm, M, N, K, "fp32", workspace_bytes=1 << 62).workspace_bytes
    x = torch.zeros((M, K), device="cuda")
    w = torch.zeros((N, K), device="cuda")
    y = torch.zeros((M, N), device="cuda")
    if need <= tll.STATIC_SCRATCH_BYTES:
        pytest.skip(f"on {sm} SMs this shape's split fits the array ({need} bytes)")
    y0 = y.clone()
    assert _static(lib, x, w, None, y, tll.EPI_NONE) == tll.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(y, y0)  # nothing was launched


def test_static_scratch_inside_graph_capture():
    """What the entry exists for: after one eager call, the call can be
    captured in a CUDA graph (nothing is allocated while capturing), and each
    replay recomputes the layer (checked against the oracle)."""
    lib = tll.library()
    layer = si.GPT2_M128_FP32[3]  # fc2: a split through the static array
    X, W, b = si.make_inputs(layer)
    x, w, bias = torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda()
    y = torch.empty((layer.M, layer.N), device="cuda")
    assert _static(lib, x, w, bias, y, tll.EPI_NONE) == tll.OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert _static(lib, x, w, bias, y, tll.EPI_NONE) == tll.OK
    ref = oracle.linear(X, W, b)
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert oracle.rel_err(y.double().cpu().numpy(), ref) <= oracle.TOL[si.PREC_FP32]
