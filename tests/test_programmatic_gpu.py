"""Programmatic launch (the default): a call's CTAs may start while the
previous kernel on the stream runs and ask the L2 for their operands, but
read nothing before griddepcontrol.wait. These tests check that this changes
no result: the same bits with the option on and off, chains of calls (each
reading the previous call's output) queued back to back equal the same calls
made one at a time, and a call right after a framework kernel that rewrites
its X sees the new X."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll

pytestmark = pytest.mark.gpu

BF16, TF32, FP32 = si.PREC_BF16, si.PREC_TF32, si.PREC_FP32
NAME = {BF16: "bf16", TF32: "tf32", FP32: "fp32"}
# one square layer per kernel family (N = K, so a call can read the previous call's output)
LAYERS = [
    si.Layer("skinny", 16, 4096, 4096, BF16, bias=True),
    si.Layer("tc_bf16", 512, 1024, 1024, BF16, si.EPI_GELU, bias=True),
    si.Layer("tc_tf32", 384, 768, 768, TF32, bias=True, x_dist="uniform"),
    si.Layer("ffma", 128, 768, 768, FP32, si.EPI_GELU, bias=True),
    si.Layer("gemv", 4, 512, 512, FP32, bias=True),
]


def _dev(a, prec):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if prec == BF16 else t


@pytest.mark.parametrize("layer", LAYERS, ids=lambda l: l.name)
def test_same_bits_with_and_without_programmatic_launch(layer):
    X, W, b = si.make_inputs(layer)
    x, w, bias = _dev(X, layer.precision), _dev(W, layer.precision), torch.from_numpy(b).cuda()
    epi = "gelu" if layer.epilogue else "none"
    outs = []
    for prog in (1, 0):
        ctx = tll.Context(0)
        ctx.set_option(tll.OPT_PROGRAMMATIC_LAUNCH, prog)
        outs.append(tll.forward(x, w, bias, epilogue=epi, precision=NAME[layer.precision], ctx=ctx))
        torch.cuda.synchronize()
        ctx.check()
    assert torch.equal(outs[0], outs[1])
    ref = oracle.linear(X, W, b, bool(layer.epilogue))
    assert oracle.rel_err(outs[0].double().cpu().numpy(), ref) <= oracle.TOL[layer.precision]


@pytest.mark.parametrize("layer", LAYERS, ids=lambda l: l.name)
def test_chain_queued_equals_one_at_a_time(layer):
    """Eight layers in a row, each reading the previous layer's output and a
    different W, queued without synchronisation (programmatic launch, nothing
    read early) against the same calls with a device synchronisation between
    them."""
    X, _, b = si.make_inputs(layer)
    prec = layer.precision
    ws = [_dev(si.round_bf16(si.normal(70 + i, 2, (layer.N, layer.K), 0.0, 0.02)) if prec == BF16 else
               si.normal(70 + i, 2, (layer.N, layer.K), 0.0, 0.02 if prec != TF32 else 0.04), prec) for i in range(3)]
    bias = torch.from_numpy(b).cuda()
    epi = "gelu" if layer.epilogue else "none"
    ctx = tll.Context(0)
    x0 = _dev(X, prec)
    chain = [x0]
    for i in range(8):
        chain.append(tll.forward(chain[-1], ws[i % 3], bias, epilogue=epi, precision=NAME[prec], ctx=ctx))
    torch.cuda.synchronize()
    ctx.check()
    y = x0
    for i in range(8):
        y = tll.forward(y, ws[i % 3], bias, epilogue=epi, precision=NAME[prec], ctx=ctx)
        torch.cuda.synchronize()
        assert torch.equal(y, chain[i + 1]), i
    # and the first link against the oracle
    ref = oracle.linear(X, ws[0].float().cpu().numpy(), b, bool(layer.epilogue))
    assert oracle.rel_err(chain[1].double().cpu().numpy(), ref) <= oracle.TOL[prec]


@pytest.mark.parametrize("layer", LAYERS, ids=lambda l: l.name)
def test_call_sees_a_framework_kernels_write(layer):
    """A torch kernel rewrites X (and the bias) right before the call on the
    same stream; the call, launched as a programmatic dependent of it, must
    use the new values."""
    X, W, b = si.make_inputs(layer)
    prec = layer.precision
    x, w, bias = _dev(X, prec), _dev(W, prec), torch.from_numpy(b).cuda()
    ctx = tll.Context(0)
    epi = "gelu" if layer.epilogue else "none"
    tll.forward(x, w, bias, epilogue=epi, precision=NAME[prec], ctx=ctx)  # warm: the stream's last call
    for _ in range(3):
        x.mul_(-1.0)       # framework kernels on the same stream, just before the call
        bias.add_(0.5)
        y = tll.forward(x, w, bias, epilogue=epi, precision=NAME[prec], ctx=ctx)
    torch.cuda.synchronize()
    ctx.check()
    ref = oracle.linear(-X, W, b + 1.5, bool(layer.epilogue))
    assert oracle.rel_err(y.double().cpu().numpy(), ref) <= oracle.TOL[prec]
