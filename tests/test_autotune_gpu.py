"""Measured dispatch: installed plans (lin_set_plan_override) and the
autotuner that picks them. lin_forward must run an installed plan for its
exact call signature only, keep parity with the oracle under it, and refuse
a plan that cannot run the shape without losing the entry it had."""
import json

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll
from transformer_linear_layer_gb300 import autotune
from gpu_util import check_layer, run

pytestmark = pytest.mark.gpu

BF16, TF32, FP32 = si.PREC_BF16, si.PREC_TF32, si.PREC_FP32


def _same(a, b):
    return autotune._plan_key(a) == autotune._plan_key(b)


@pytest.fixture
def ctx():
    c = tll.Context(0)
    yield c
    c.close()


def test_installed_plan_is_used_and_removed(ctx):
    layer = si.Layer("ovr_bf16", 256, 768, 768, BF16, si.EPI_GELU, bias=True)
    default = ctx.plan(256, 768, 768, "bf16", "gelu")
    alt = next(p for p in autotune.candidates(ctx.sm_count, 256, 768, 768, "bf16", ctx.workspace_bytes)
               if not _same(p, default))
    ctx.set_override(256, 768, 768, "bf16", "gelu", alt)
    check_layer(layer, ctx=ctx)
    assert _same(ctx.last_plan(), alt)
    # another epilogue is another call signature: the built-in table runs it
    check_layer(si.Layer("ovr_bf16_noact", 256, 768, 768, BF16, bias=True), ctx=ctx)
    assert not _same(ctx.last_plan(), alt)
    ctx.set_override(256, 768, 768, "bf16", "gelu", None)
    check_layer(layer, ctx=ctx)
    assert _same(ctx.last_plan(), default)


def test_refused_plan_keeps_the_entry(ctx):
    M, N, K = 130, 520, 2200
    good = tll.plan_make(ctx.sm_count, tll.KERNEL_FFMA, 0, 3, M, N, K, "fp32")
    ctx.set_override(M, N, K, "fp32", "none", good)
    bad = tll.plan_make(ctx.sm_count, tll.KERNEL_TC, 0, 0, M, N, K, "tf32")  # a tensor-core plan for fp32
    with pytest.raises(tll.LinError):
        ctx.set_override(M, N, K, "fp32", "none", bad)
    small = tll.plan_make(ctx.sm_count, tll.KERNEL_FFMA, 0, 1, 64, 64, 64, "fp32")  # grid for another shape
    with pytest.raises(tll.LinError):
        ctx.set_override(M, N, K, "fp32", "none", small)
    check_layer(si.Layer("ovr_fp32", M, N, K, FP32, bias=True), ctx=ctx)
    assert _same(ctx.last_plan(), good)
    ctx.clear_overrides()
    check_layer(si.Layer("ovr_fp32", M, N, K, FP32, bias=True), ctx=ctx)
    # the built-in table again (its split may be narrowed for a call that overlaps the previous one)
    last = ctx.last_plan()
    assert not _same(last, good) and last.kernel == tll.KERNEL_FFMA


@pytest.mark.parametrize("M,N,K,precision,epi", [
    (128, 2304, 768, BF16, si.EPI_NONE),
    (8, 3072, 768, BF16, si.EPI_GELU),
    (128, 768, 3072, FP32, si.EPI_NONE),
    (512, 1024, 1024, TF32, si.EPI_GELU),
])
def test_autotune_keeps_parity(ctx, M, N, K, precision, epi):
    """Tune one shape, then the tuned lin_forward still matches the oracle and
    runs the reported winner (or the built-in plan when nothing won)."""
    pname = {BF16: "bf16", TF32: "tf32", FP32: "fp32"}[precision]
    ename = "gelu" if epi == si.EPI_GELU else "none"
    (rep,) = autotune.autotune(ctx, [(M, N, K, pname, ename)], rounds=3, reps=8)
    assert rep["incumbent_us"] > 0 and rep["roofline_floor_us"] > 0
    assert len(rep["screened"]) >= 1
    assert rep["incumbent_us"] >= 0.5 * rep["roofline_floor_us"]  # a call cannot beat the roofline by 2x
    check_layer(si.Layer("tuned", M, N, K, precision, epi, bias=True), ctx=ctx)
    if rep["winner"] is None:
        # the built-in table ran (its plan, or the same family narrowed for a back-to-back call)
        assert ctx.last_plan().kernel == ctx.plan(M, N, K, pname, ename).kernel
    else:
        assert rep["winner_ratio"] < 1.0
        assert ctx.last_plan().as_dict() == rep["winner"]


def test_save_and_load_round_trip(ctx, tmp_path):
    M, N, K = 64, 512, 1024
    win = tll.plan_make(ctx.sm_count, tll.KERNEL_FFMA, 0, 3, M, N, K, "fp32")
    reports = [{"shape": [M, N, K], "precision": "fp32", "epilogue": "none", "winner": win.as_dict()},
               {"shape": [1, 2, 3], "precision": "fp32", "epilogue": "none", "winner": None}]
    path = tmp_path / "plans.json"
    autotune.save(reports, str(path))
    assert len(json.loads(path.read_text())) == 1
    fresh = tll.Context(0)
    try:
        assert autotune.load(fresh, str(path)) == 1
        X, W, b = si.make_inputs(si.Layer("rt", M, N, K, FP32, bias=True))
        y = run(X, W, b, FP32, ctx=fresh)
        assert oracle.rel_err(y, oracle.linear(X, W, b, False)) <= oracle.TOL[FP32]
        assert _same(fresh.last_plan(), win)
    finally:
        fresh.close()


def test_fixed_plans_give_history_independent_bits(ctx):
    """With adaptive plans off, a call gives the same bits alone and right
    after an independent call; with them on (the default) the overlapping
    call may drop its K split: other rounding, same tolerance."""
    import torch

    M, N, K = 128, 2304, 768
    layer = si.Layer("hist", M, N, K, FP32, bias=True)
    X, W, b = si.make_inputs(layer)
    x, w, bias = (torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda())
    w2 = w.clone()
    ref = oracle.linear(X, W, b, False)
    s = torch.cuda.Stream()

    def pair():
        """(isolated call's Y, plan), (back-to-back call's Y, plan)."""
        with torch.cuda.stream(s):
            ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)
            y1 = tll.forward(x, w, bias, precision="fp32", ctx=ctx)
            p1 = ctx.last_plan()
            ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_ALL)
            tll.forward(x, w2, bias, precision="fp32", ctx=ctx, out=torch.empty_like(y1))
            y2 = tll.forward(x, w, bias, precision="fp32", ctx=ctx)
            p2 = ctx.last_plan()
        s.synchronize()
        ctx.check(s)
        return (y1, p1), (y2, p2)

    (y1, p1), (y2, p2) = pair()
    assert p1.splits > 1 and p2.splits < p1.splits  # adaptive plans drop the split back to back
    for y in (y1, y2):
        assert oracle.rel_err(y.double().cpu().numpy(), ref) <= oracle.TOL[FP32]
    ctx.set_option(tll.OPT_ADAPTIVE_PLANS, 0)
    try:
        (y1, p1), (y2, p2) = pair()
    finally:
        ctx.set_option(tll.OPT_ADAPTIVE_PLANS, 1)
        ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)
    assert _same(p1, p2) and torch.equal(y1, y2)
