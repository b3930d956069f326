"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances (max|Y - Y_ref| / max|Y_ref|): 1e-5 for fp32, 5e-3 for TF32,
1e-2 for bf16 inputs; exact-arithmetic cases (permutation weights, small
integer inputs) must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll
from gpu_util import PREC_NAME, check_layer, device_inputs, run

pytestmark = pytest.mark.gpu

BF16, TF32, FP32 = si.PREC_BF16, si.PREC_TF32, si.PREC_FP32


@pytest.fixture(scope="module")
def ctx():
    return tll.default_context(0)


@pytest.fixture(scope="module", autouse=True)
def _early_start_all():
    """These tests run back-to-back library calls only, so the programmatic
    early start (inputs read before the previous kernel finishes) is safe and
    is what they exercise; the library's default is off."""
    c = tll.default_context(0)
    c.set_option(tll.OPT_EARLY_START, tll.EARLY_ALL)
    yield
    c.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)


def all_plans(ctx, M, N, K, precision):
    """Every kernel family / variant that can run this shape, plus split choices."""
    plans = []
    sm = ctx.sm_count
    if precision == BF16 and M <= 16:
        for v in range(5):
            for s in (0, 1, 2, 8):
                plans.append(tll.plan_make(sm, tll.KERNEL_SKINNY, v, s, M, N, K, "bf16"))
    if precision in (BF16, TF32):
        for v in range(6):  # 3-5: SM pairs (2-CTA clusters, cta_group::2 MMAs on 256-row tiles)
            for width in (0, 1, 3):  # persistent CTAs: one per SM, or few CTAs walking many tiles
                plans.append(tll.plan_make(sm, tll.KERNEL_TC, v, width, M, N, K, PREC_NAME[precision]))
        for v in range(3):  # stream-K with few CTAs, so that tiles are cut between CTAs
            for ctas in (2, 3, 5):
                try:
                    plans.append(tll.plan_make(sm, tll.KERNEL_TC, v, -ctas, M, N, K, PREC_NAME[precision]))
                except tll.LinError:  # fewer tiles than CTAs: no stream-K plan
                    pass
    if precision == FP32:
        for v in range(4):  # 128x128, 64x64, 128x128 with K steps of 64, 128x64
            for s in (1, 0, 3):
                plans.append(tll.plan_make(sm, tll.KERNEL_FFMA, v, s, M, N, K, "fp32"))
    if (precision in (FP32, TF32) and M <= 8) or (precision == BF16 and M <= 4):
        for ctas in (0, 3):  # as many CTAs as fit, or a few walking many rows of W
            try:
                plans.append(tll.plan_make(sm, tll.KERNEL_GEMV, 0, ctas, M, N, K, PREC_NAME[precision]))
            except tll.LinError:  # X does not fit in shared memory
                pass
    return plans


# ---------------------------------------------------------------- exact cases

@pytest.mark.parametrize("precision", [BF16, TF32, FP32])
@pytest.mark.parametrize("M,N,K", [(16, 96, 96), (200, 136, 136), (5, 72, 72)])
def test_permutation_weights_exact(ctx, precision, M, N, K):
    """W a permutation matrix (N = K): Y = X[:, p] exactly, on every kernel.
    Pins operand roles and the smem/TMEM layouts (a one-hot probe per column)."""
    p = (np.arange(K) * 7 + 3) % K
    W = np.zeros((N, K), np.float32)
    W[np.arange(N), p[:N]] = 1.0
    X = si.uniform_pm1(3, M, (M, K))
    if precision == BF16:
        X = si.round_bf16(X)
    for plan in all_plans(ctx, M, N, K, precision):
        y = run(X, W, None, precision, plan=plan, ctx=ctx)
        expect = X[:, p[:N]].astype(np.float64)
        if precision == TF32:
            # the tensor core multiplies the TF32 part of X (1 x value keeps 10 mantissa bits)
            assert np.max(np.abs(y - expect)) <= 2.0 ** -10 * np.max(np.abs(expect)), plan
            continue
        assert np.array_equal(y, expect), f"plan {plan}"


@pytest.mark.parametrize("precision", [BF16, TF32, FP32])
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (1, 40, 64), (129, 264, 200), (300, 520, 1024)])
def test_small_integers_bitwise(ctx, precision, M, N, K):
    """Integer inputs in [-4, 4]: every product and partial sum is exact, so the
    GPU must equal the oracle bit for bit (bf16 output: the oracle's value
    rounded to nearest-even bf16)."""
    layer = si.Layer("ints", M, N, K, precision, bias=True, x_dist="ints")
    X, W, b = si.make_inputs(layer)
    ref = oracle.linear(X, W, b)
    if precision == BF16:
        ref = si.round_bf16(ref.astype(np.float32)).astype(np.float64)
    for plan in all_plans(ctx, M, N, K, precision):
        y = run(X, W, b, precision, plan=plan, ctx=ctx)
        assert np.array_equal(y, ref), f"plan {plan}: max diff {np.max(np.abs(y - ref))}"


# ------------------------------------------------------------ the workloads

def test_square_256_fp32(ctx):
    layer = si.SQUARE_256_FP32
    for plan in [None] + all_plans(ctx, 256, 256, 256, FP32):
        check_layer(layer, plan=plan, ctx=ctx)


def test_skinny_m16_4096_every_variant(ctx):
    layer = si.SKINNY_16x4096
    for plan in [None] + all_plans(ctx, 16, 4096, 4096, BF16):
        check_layer(layer, plan=plan, ctx=ctx)


@pytest.mark.parametrize("layer", si.GPT2_M128_FP32, ids=lambda l: l.name)
def test_gpt2_m128_fp32(ctx, layer):
    check_layer(layer, ctx=ctx)


@pytest.mark.parametrize("layer", [si.SQUARE_4096_FP32, si.SQUARE_4096_TF32], ids=lambda l: l.name)
def test_square_4096_full(layer):
    """All 4096 x 4096 outputs against the oracle."""
    check_layer(layer)


@pytest.mark.parametrize("layer", si.GPT2_M8192_BF16, ids=lambda l: l.name)
def test_gpt2_m8192_bf16_full(layer):
    """All M x N outputs of every batched GPT-2 layer against the oracle, the
    LM head's 8192 x 50257 included (every tile of the persistent schedule,
    its last rounds and the ragged N tail)."""
    check_layer(layer)


@pytest.mark.parametrize("precision", [BF16, TF32])
def test_tc_midsize_full(ctx, precision):
    """Several tiles in each direction and ragged tails, full comparison."""
    for M, N, K in [(384, 640, 768), (257, 1000, 320), (131, 50257 % 1024 + 512, 96)]:
        layer = si.Layer("tc_mid", M, N, K, precision, si.EPI_GELU, bias=True)
        for plan in all_plans(ctx, M, N, K, precision):
            check_layer(layer, plan=plan, ctx=ctx)


@pytest.mark.parametrize("M,N,K,precision", [(8192, 768, 768, BF16), (8192, 768, 3072, BF16),
                                             (2560, 2560, 512, BF16), (4352, 1280, 512, TF32)])
def test_tail_split(M, N, K, precision):
    """More tiles than SMs with a ragged last round, through an explicit plan
    (the built-in table runs such tiles whole): whole rounds of tiles, then
    the remaining tiles split in K and added in split order (on its own context
    and stream). Every output against the oracle, bitwise repeatable."""
    c = tll.Context(0)
    plan = tll.plan_make(c.sm_count, tll.KERNEL_TC, 0, 0, M, N, K, PREC_NAME[precision])
    tiles = ((M + 127) // 128) * ((N + plan.bn - 1) // plan.bn)
    rest = tiles - tiles // plan.grid_x * plan.grid_x
    nkb = (K * (2 if precision == BF16 else 4) + 127) // 128
    splits = min(plan.grid_x // rest, nkb // 4, 16)
    assert tiles > plan.grid_x and 0 < 2 * rest <= plan.grid_x and splits > 1, (tiles, rest, splits)
    plan.grid_z = splits
    plan.workspace_bytes = (64 << 10) + rest * splits * 128 * plan.bn * 4
    assert tll.plan_check(plan, M, N, K, PREC_NAME[precision], c.workspace_bytes) == tll.OK
    layer = si.Layer("tail_split", M, N, K, precision, si.EPI_GELU, bias=True,
                     x_dist="uniform" if precision == TF32 else "normal")
    X, W, b = si.make_inputs(layer)
    st = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        with torch.cuda.stream(st):
            x, w, bias = device_inputs(X, W, b, precision)
            outs.append(tll.forward_plan(plan, x, w, bias, epilogue="gelu", precision=PREC_NAME[precision], ctx=c,
                                         stream=st))
        st.synchronize()
    c.check(st)
    assert c.last_plan().grid_z == plan.grid_z
    assert torch.equal(outs[0], outs[1])
    ref = oracle.linear(X, W, b, True)
    assert oracle.rel_err(outs[0].double().cpu().numpy(), ref) <= oracle.TOL[precision]
    c.close()


@pytest.mark.parametrize("r", range(1, 8))
def test_unaligned_rows_bf16(ctx, r):
    """bf16 Y with rows that are not 16-byte aligned (N = 8q + r): the row
    segments of a chunk start at every misalignment, and the vector-store
    epilogue must write each element once and nothing beyond the row, on the
    single-CTA and SM-pair 256-column tiles (several tiles, a ragged M and the
    matrix's last column chunk), with and without GELU."""
    N = 1024 + 256 + r
    for M, K, epi in ((300, 256, si.EPI_GELU), (131, 320, si.EPI_NONE)):
        layer = si.Layer("unaligned", M, N, K, BF16, epi, bias=True)
        for v in (0, 3):
            plan = tll.plan_make(ctx.sm_count, tll.KERNEL_TC, v, 0, M, N, K, "bf16")
            check_layer(layer, plan=plan, ctx=ctx)
    # the neighbours of Y are untouched
    X, W, b = si.make_inputs(si.Layer("unaligned_guard", 130, N, 256, BF16, bias=True))
    x, w, bias = device_inputs(X, W, b, BF16)
    big = torch.full((130 * N + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = big[16:16 + 130 * N].view(130, N)  # 32-byte offset: 16-byte aligned base
    tll.forward(x, w, bias, precision="bf16", out=y, ctx=ctx)
    torch.cuda.synchronize()
    assert bool((big[:16] == 7.0).all()) and bool((big[16 + 130 * N:] == 7.0).all())
    ref = oracle.linear(X, W, b)
    assert oracle.rel_err(y.double().cpu().numpy(), ref) <= oracle.TOL[BF16]


def test_unaligned_rows_bf16_each_element_written_once(ctx):
    """The odd-row store path (16-byte blocks of each row's segment, the block
    shared by two chunks of a warp completed from the previous chunk) against
    the element-by-element path of the same kernel (Y at a 2-byte offset): the
    same bits, and no output left unwritten (Y starts as NaN), for every row
    misalignment, ragged M and a partial last chunk."""
    for r in range(1, 8):
        N = 1024 + 256 + 32 + r
        M, K = 260, 192
        X, W, b = si.make_inputs(si.Layer("unaligned_once", M, N, K, BF16, si.EPI_GELU, bias=True))
        x, w, bias = device_inputs(X, W, b, BF16)
        for v in (0, 3):
            plan = tll.plan_make(ctx.sm_count, tll.KERNEL_TC, v, 0, M, N, K, "bf16")
            y_vec = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            flat = torch.full((M * N + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
            y_el = flat[1:1 + M * N].view(M, N)  # 2-byte offset: the element-by-element path
            tll.forward_plan(plan, x, w, bias, epilogue="gelu", precision="bf16", out=y_vec, ctx=ctx)
            tll.forward_plan(plan, x, w, bias, epilogue="gelu", precision="bf16", out=y_el, ctx=ctx)
            torch.cuda.synchronize()
            ctx.check()
            assert not bool(torch.isnan(y_vec).any()), f"N={N} variant {v}: an output was not written"
            assert torch.equal(y_vec, y_el), f"N={N} variant {v}"
            assert oracle.rel_err(y_vec.double().cpu().numpy(), oracle.linear(X, W, b, True)) <= oracle.TOL[BF16]


# ------------------------------------------------------------- edge shapes

@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 127, 129])
def test_edge_rows_bf16(ctx, M):
    check_layer(si.Layer("edge", M, 1000, 520, BF16, si.EPI_GELU, bias=True), ctx=ctx)


@pytest.mark.parametrize("M", [1, 3, 63, 65, 127, 129])
def test_edge_rows_fp32(ctx, M):
    check_layer(si.Layer("edge", M, 333, 132, FP32, si.EPI_GELU, bias=True), ctx=ctx)


@pytest.mark.parametrize("precision,K", [(BF16, 8), (BF16, 40), (BF16, 4104), (TF32, 4), (TF32, 36), (FP32, 4),
                                         (FP32, 20)])
def test_k_tails(ctx, precision, K):
    for M in (16, 160):
        layer = si.Layer("ktail", M, 200, K, precision, bias=True)
        for plan in [None] + all_plans(ctx, M, 200, K, precision):
            check_layer(layer, plan=plan, ctx=ctx)


@pytest.mark.parametrize("precision", [BF16, TF32, FP32])
def test_k_zero_gives_activation_of_bias(ctx, precision):
    M, N = 7, 33
    b = si.normal(1, 1, (N,), 0.0, 1.0)
    x, w, bias = device_inputs(np.zeros((M, 0), np.float32), np.zeros((N, 0), np.float32), b, precision)
    y = tll.forward(x, w, bias, epilogue="gelu", precision=PREC_NAME[precision])
    ref = oracle.linear(np.zeros((M, 0), np.float32), np.zeros((N, 0), np.float32), b, True)
    assert oracle.rel_err(y.float().cpu().numpy(), ref) <= oracle.TOL[precision]


def test_empty_m_and_n(ctx):
    x = torch.zeros((0, 64), device="cuda", dtype=torch.bfloat16)
    w = torch.zeros((32, 64), device="cuda", dtype=torch.bfloat16)
    assert tll.forward(x, w).shape == (0, 32)
    x = torch.zeros((4, 64), device="cuda", dtype=torch.bfloat16)
    w = torch.zeros((0, 64), device="cuda", dtype=torch.bfloat16)
    assert tll.forward(x, w).shape == (4, 0)


# ------------------------------------------------------------- properties

@pytest.mark.parametrize("precision,M,N,K", [(BF16, 16, 4096, 4096), (FP32, 128, 768, 3072), (BF16, 384, 512, 768),
                                             (TF32, 256, 384, 512)])
def test_bitwise_repeatable(ctx, precision, M, N, K):
    """Split-K and all: two runs give identical bits (fixed-order reduction)."""
    X, W, b = si.make_inputs(si.Layer("rep", M, N, K, precision, bias=True))
    y1 = run(X, W, b, precision, ctx=ctx)
    y2 = run(X, W, b, precision, ctx=ctx)
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("precision,M,N,K", [(BF16, 16, 1024, 1024), (FP32, 128, 768, 768), (BF16, 256, 512, 256),
                                             (TF32, 256, 256, 128)])
def test_identical_rows_identical_outputs(ctx, precision, M, N, K):
    """Every row of X the same: every row of Y must be the same, bitwise (no
    leak between rows of a batch)."""
    X1, W, b = si.make_inputs(si.Layer("rows", 1, N, K, precision, bias=True))
    X = np.repeat(X1, M, axis=0)
    y = run(X, W, b, precision, ctx=ctx)
    assert np.array_equal(y, np.repeat(y[:1], M, axis=0))


@pytest.mark.parametrize("precision,M,N,K", [(BF16, 16, 300, 256), (BF16, 140, 300, 256), (FP32, 70, 300, 256),
                                             (TF32, 140, 300, 256)])
def test_no_writes_outside_y(ctx, precision, M, N, K):
    """Canary: Y sits inside a larger buffer filled with a sentinel; only the
    M x N window may change."""
    X, W, b = si.make_inputs(si.Layer("canary", M, N, K, precision, bias=True))
    x, w, bias = device_inputs(X, W, b, precision)
    dt = torch.bfloat16 if precision == BF16 else torch.float32
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345.0, device="cuda", dtype=dt)
    out = buf[pad:pad + M * N].view(M, N)
    tll.forward(x, w, bias, precision=PREC_NAME[precision], out=out)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == 12345.0).all()) and bool((buf[pad + M * N:] == 12345.0).all())
    ref = oracle.linear(X, W, b)
    assert oracle.rel_err(out.float().cpu().numpy(), ref) <= oracle.TOL[precision]


# ------------------------------------------------------------ error paths

def test_status_codes(ctx):
    x = torch.zeros((16, 64), device="cuda", dtype=torch.bfloat16)
    w = torch.zeros((32, 64), device="cuda", dtype=torch.bfloat16)
    y = torch.empty((16, 32), device="cuda", dtype=torch.bfloat16)
    s = torch.cuda.current_stream().cuda_stream
    # misaligned X (2-byte offset)
    xb = torch.zeros((16 * 64 + 8,), device="cuda", dtype=torch.bfloat16)
    assert ctx.forward_ptr(16, 32, 64, xb.data_ptr() + 2, w.data_ptr(), None, y.data_ptr(), 0, 2, s) == tll.ERR_ALIGN
    # K * 2 bytes not a multiple of 16
    assert ctx.forward_ptr(16, 32, 60, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 0, 2, s) == tll.ERR_ALIGN
    # Y overlapping X
    assert ctx.forward_ptr(16, 32, 64, x.data_ptr(), w.data_ptr(), None, x.data_ptr(), 0, 2, s) == tll.ERR_ARG
    # bad enums, negative sizes, NULL pointers
    assert ctx.forward_ptr(16, 32, 64, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 7, 2, s) == tll.ERR_ARG
    assert ctx.forward_ptr(-1, 32, 64, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 0, 2, s) == tll.ERR_ARG
    assert ctx.forward_ptr(16, 32, 64, None, w.data_ptr(), None, y.data_ptr(), 0, 2, s) == tll.ERR_ARG
    # a plan for another kernel family or shape
    plan = tll.plan_make(ctx.sm_count, tll.KERNEL_FFMA, 0, 1, 16, 32, 64, "fp32")
    assert ctx.forward_plan_ptr(plan, 16, 32, 64, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 0, 2,
                                s) == tll.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    ctx.check()


def test_workspace_limit():
    small = tll.Context(0, workspace_bytes=4096)
    M, N, K = 128, 768, 3072
    x = torch.zeros((M, K), device="cuda", dtype=torch.float32)
    w = torch.zeros((N, K), device="cuda", dtype=torch.float32)
    # the dispatch table fits the split to the workspace (here: no split)...
    assert small.plan(M, N, K, "fp32").splits == 1
    tll.forward(x, w, ctx=small)
    # ...an explicit plan that needs more is refused
    plan = tll.plan_make(small.sm_count, tll.KERNEL_FFMA, 1, 6, M, N, K, "fp32")
    assert plan.workspace_bytes > 4096
    y = torch.empty((M, N), device="cuda", dtype=torch.float32)
    rc = small.forward_plan_ptr(plan, M, N, K, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), 0, 0,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == tll.ERR_WORKSPACE
    small.check()
    small.close()


@pytest.mark.parametrize("M", [16, 256])
def test_back_to_back_calls_chain_through_outputs(ctx, M):
    """Layer i+1 reads layer i's output (X = previous Y) and, in a second chain,
    its weight is the previous output: both must match running the layers one
    at a time (the early start must wait for X and must not prefetch a W that
    the previous call writes). M = 16: skinny kernel; M = 256: tcgen05 kernel."""
    N = 512
    X0, W, b = si.make_inputs(si.Layer("chain", M, N, N, BF16, bias=True))
    x0, w, bias = device_inputs(X0, W, b, BF16)
    outs = [x0]
    for _ in range(6):
        outs.append(tll.forward(outs[-1], w, bias, precision="bf16"))
    torch.cuda.synchronize()
    ref = x0
    for i in range(6):
        ref = tll.forward(ref, w, bias, precision="bf16")
        torch.cuda.synchronize()
        assert torch.equal(ref, outs[i + 1])
    # W of call i+1 = Y of call i (N x N square so the shapes line up)
    wsq = w.clone()
    y1 = tll.forward(x0[:16], wsq, None, precision="bf16")          # 16 x 512
    big = torch.empty((N, N), device="cuda", dtype=torch.bfloat16)
    big[:16] = 0
    tll.forward(wsq, wsq, None, precision="bf16", out=big)           # writes big (512 x 512)
    y2 = tll.forward(x0, big, None, precision="bf16")                # reads big as W right after
    torch.cuda.synchronize()
    y2_ref = tll.forward(x0, big.clone(), None, precision="bf16")
    torch.cuda.synchronize()
    assert torch.equal(y2, y2_ref) and y1.shape == (16, N)
    # and the bias written by the previous call
    bsrc = torch.zeros((2, N), device="cuda", dtype=torch.float32)
    xf = torch.from_numpy(si.normal(9, 1, (2, 64))).cuda()
    wf = torch.from_numpy(si.normal(9, 2, (N, 64), 0.0, 0.1)).cuda()
    tll.forward(xf, wf, None, precision="fp32", out=bsrc)             # writes the bias
    y3 = tll.forward(x0, w, bsrc[1], precision="bf16")
    torch.cuda.synchronize()
    y3_ref = tll.forward(x0, w, bsrc[1].clone(), precision="bf16")
    torch.cuda.synchronize()
    assert torch.equal(y3, y3_ref)


@pytest.mark.parametrize("precision", [BF16, TF32])
def test_stream_k_cut_tiles(ctx, precision):
    """Stream-K plans whose shares cut tiles at every kind of place (within
    the first, middle and last K stages, one K stage, ragged K) against the
    oracle, full comparison; and bitwise repeatable."""
    for M, N, K, ctas in [(384, 640, 768, 4), (384, 640, 768, 7), (257, 1000, 320, 5), (256, 512, 136, 3),
                          (640, 256, 1024, 4)]:
        layer = si.Layer("sk", M, N, K, precision, si.EPI_GELU, bias=True)
        X, W, b = si.make_inputs(layer)
        ref = oracle.linear(X, W, b, True)
        for v in range(3):
            try:
                plan = tll.plan_make(ctx.sm_count, tll.KERNEL_TC, v, -ctas, M, N, K, PREC_NAME[precision])
            except tll.LinError:
                continue
            assert plan.splits == 2
            y = run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx)
            assert oracle.rel_err(y, ref) <= oracle.TOL[precision], (M, N, K, ctas, v)
            y2 = run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx)
            assert np.array_equal(y, y2)


@pytest.mark.parametrize("precision,M,N,K", [(BF16, 256, 768, 4096), (BF16, 200, 300, 4104), (TF32, 130, 520, 2200),
                                             (BF16, 512, 512, 16384), (BF16, 128, 128, 8192)])
def test_tc_k_split(ctx, precision, M, N, K):
    """Few output tiles and a long K: the dispatch table splits K (grid_z);
    each split's region goes through the workspace and the last split adds
    them in order. Full comparison with the oracle, bias and GELU, ragged
    tails; bitwise repeatable; and the split plan's calls back to back
    through the shared workspace equal the same calls one at a time."""
    plan = ctx.plan(M, N, K, PREC_NAME[precision], "gelu")
    assert tll.KERNEL_NAMES[plan.kernel] == "tc" and plan.grid_z > 1, plan
    layer = si.Layer("ksplit", M, N, K, precision, si.EPI_GELU, bias=True)
    X, W, b = si.make_inputs(layer)
    y = run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx)
    assert oracle.rel_err(y, oracle.linear(X, W, b, True)) <= oracle.TOL[precision]
    assert np.array_equal(y, run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx))
    x, w, bias = device_inputs(X, W, b, precision)
    ws = [w, w * 2, w * 3]
    prec = PREC_NAME[precision]
    outs = [tll.forward_plan(plan, x, ws[i % 3], bias, epilogue="gelu", precision=prec, ctx=ctx) for i in range(6)]
    torch.cuda.synchronize()
    for i in range(6):
        ref = tll.forward_plan(plan, x, ws[i % 3], bias, epilogue="gelu", precision=prec, ctx=ctx)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref), i
    # the public call: the same bits (split kept for a call with no
    # independent predecessor, dropped for one with it; both agree with the oracle)
    y2 = tll.forward(x, w, bias, epilogue="gelu", precision=prec, ctx=ctx)
    torch.cuda.synchronize()
    assert oracle.rel_err(y2.float().cpu().numpy().astype(np.float64), oracle.linear(X, W, b, True)) <= \
        oracle.TOL[precision]
    ctx.check()


def test_stream_k_back_to_back(ctx):
    """Stream-K calls launched back to back overlap on the GPU (the early
    start) and share the workspace slots and flags: independent calls into
    separate outputs, and a chain X = previous Y, must equal the same calls
    made one at a time."""
    M, N, K = 2560, 2048, 2048   # 20 x 8 tiles of 128 x 256: at least one per SM
    plan = tll.plan_make(ctx.sm_count, tll.KERNEL_TC, 0, -1, M, N, K, "bf16")
    assert plan.splits == 2
    X0, _, b = si.make_inputs(si.Layer("skb2b", M, N, K, BF16, bias=True))
    x0 = torch.from_numpy(X0).cuda().to(torch.bfloat16)
    bias = torch.from_numpy(b).cuda()
    ws = [torch.from_numpy(si.round_bf16(si.normal(40 + i, 2, (N, K), 0.0, 0.02))).to(torch.bfloat16).cuda()
          for i in range(3)]

    def call(x, w):
        return tll.forward_plan(plan, x, w, bias, precision="bf16", ctx=ctx)

    outs = [call(x0, ws[i % 3]) for i in range(8)]
    torch.cuda.synchronize()
    for i in range(8):
        ref = call(x0, ws[i % 3])
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref), i
    chain = [x0]
    for i in range(5):
        chain.append(call(chain[-1], ws[i % 3]))
    torch.cuda.synchronize()
    ref = x0
    for i in range(5):
        ref = call(ref, ws[i % 3])
        torch.cuda.synchronize()
        assert torch.equal(ref, chain[i + 1]), i
    ctx.check()
    # and every output against the oracle
    got = outs[0].float().cpu().numpy().astype(np.float64)
    W0 = ws[0].float().cpu().numpy()
    assert oracle.rel_err(got, oracle.linear(X0, W0, b, False)) <= oracle.TOL[BF16]


@pytest.mark.parametrize("N,K", [(768, 768), (768, 3072)])
def test_ffma_back_to_back(ctx, N, K):
    """fp32 split-K calls launched back to back (the early start) share the
    workspace partial sums and tile counters: independent calls into separate
    outputs, and a chain X = previous Y (N = K), must equal the same calls made
    one at a time. Adaptive plans are off, so that every call takes the
    table's split plan whatever precedes it (with them on, a call's split may
    depend on whether its predecessor on the stream is independent of it)."""
    M = 128
    plan = ctx.plan(M, N, K, "fp32")
    assert plan.splits > 1
    ctx.set_option(tll.OPT_ADAPTIVE_PLANS, 0)
    try:
        _ffma_back_to_back(ctx, M, N, K)
    finally:
        ctx.set_option(tll.OPT_ADAPTIVE_PLANS, 1)


def _ffma_back_to_back(ctx, M, N, K):
    X0, _, b = si.make_inputs(si.Layer("ffb2b", M, N, K, FP32, bias=True))
    x0 = torch.from_numpy(X0).cuda()
    bias = torch.from_numpy(b).cuda()
    ws = [torch.from_numpy(si.normal(60 + i, 2, (N, K), 0.0, 0.02)).cuda() for i in range(3)]
    outs = [tll.forward(x0, ws[i % 3], bias, precision="fp32") for i in range(8)]
    torch.cuda.synchronize()
    for i in range(8):
        ref = tll.forward(x0, ws[i % 3], bias, precision="fp32")
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref), i
    if N == K:
        chain = [x0]
        for i in range(5):
            chain.append(tll.forward(chain[-1], ws[i % 3], bias, epilogue="gelu", precision="fp32"))
        torch.cuda.synchronize()
        ref = x0
        for i in range(5):
            ref = tll.forward(ref, ws[i % 3], bias, epilogue="gelu", precision="fp32")
            torch.cuda.synchronize()
            assert torch.equal(ref, chain[i + 1]), i
    ctx.check()
    refv = oracle.linear(X0, ws[0].cpu().numpy(), b)
    assert oracle.rel_err(outs[0].cpu().numpy().astype(np.float64), refv) <= oracle.TOL[FP32]


@pytest.mark.parametrize("precision", [FP32, TF32, BF16])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_gemv_few_rows(ctx, precision, M):
    """The one-row sites: fp32 / tf32 with M <= 8 and bf16 with one row run the
    GEMV by default (exact fp32 arithmetic; bf16 products are exact in fp32);
    bf16 with 2-4 rows runs it through an explicit plan. Ragged N and K, bias
    and GELU, against the oracle; bitwise repeatable."""
    if precision == BF16 and M > 4:
        pytest.skip("the bf16 GEMV takes at most 4 rows")
    tol = oracle.TOL[BF16] if precision == BF16 else oracle.TOL[FP32]
    for N, K in [(1000, 520), (77, 8), (2304, 768), (300, 3072)]:
        layer = si.Layer("gemv", M, N, K, precision, si.EPI_GELU, bias=True)
        X, W, b = si.make_inputs(layer)
        plan = None
        if precision == BF16 and M > 1:
            plan = tll.plan_make(ctx.sm_count, tll.KERNEL_GEMV, 0, 0, M, N, K, "bf16")
        else:
            assert tll.KERNEL_NAMES[ctx.plan(M, N, K, PREC_NAME[precision]).kernel] == "gemv"
        y = run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx)
        ref = oracle.linear(X, W, b, True)
        assert oracle.rel_err(y, ref) <= tol, (M, N, K)
        assert np.array_equal(y, run(X, W, b, precision, epilogue=si.EPI_GELU, plan=plan, ctx=ctx))


@pytest.mark.parametrize("precision", [FP32, BF16])
def test_gemv_lm_head_row(ctx, precision):
    """The last token's logits: 1 x 50257 x 768 (N odd), full compare, through
    the built-in table (GEMV for fp32, the skinny kernel for bf16) and the GEMV."""
    layer = si.Layer("logits", 1, 50257, 768, precision, bias=False)
    check_layer(layer)
    check_layer(layer, plan=tll.plan_make(ctx.sm_count, tll.KERNEL_GEMV, 0, 0, 1, 50257, 768, PREC_NAME[precision]))


def test_gemv_back_to_back_chain(ctx):
    """GEMV calls back to back: independent ones into separate outputs, and a
    chain X = previous Y, equal the same calls one at a time."""
    M, N = 4, 1024
    X0, _, b = si.make_inputs(si.Layer("gemvb2b", M, N, N, FP32, bias=True))
    x0 = torch.from_numpy(X0).cuda()
    bias = torch.from_numpy(b).cuda()
    ws = [torch.from_numpy(si.normal(70 + i, 2, (N, N), 0.0, 0.03)).cuda() for i in range(3)]
    outs = [tll.forward(x0, ws[i % 3], bias, precision="fp32") for i in range(6)]
    chain = [x0]
    for i in range(6):
        chain.append(tll.forward(chain[-1], ws[i % 3], bias, epilogue="gelu", precision="fp32"))
    torch.cuda.synchronize()
    for i in range(6):
        ref = tll.forward(x0, ws[i % 3], bias, precision="fp32")
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref), i
    ref = x0
    for i in range(6):
        ref = tll.forward(ref, ws[i % 3], bias, epilogue="gelu", precision="fp32")
        torch.cuda.synchronize()
        assert torch.equal(ref, chain[i + 1]), i
    ctx.check()


@pytest.mark.parametrize("M,precision", [(128, FP32), (1, FP32), (256, BF16), (4, BF16)])
def test_layer_captured_in_one_graph(M, precision):
    """A transformer layer's four GEMMs (qkv, proj, fc1 + GELU, fc2 reading
    fc1's output) recorded in one CUDA graph and replayed: the library makes
    no allocation and no host sync inside the calls, and the replays give the
    eager results bit for bit (and the oracle's)."""
    d = 768
    dt = torch.bfloat16 if precision == BF16 else torch.float32
    prec = PREC_NAME[precision]
    specs = [("qkv", 3 * d, d, False), ("proj", d, d, False), ("fc1", 4 * d, d, True), ("fc2", d, 4 * d, False)]
    inputs = {}
    for i, (name, N, K, gelu) in enumerate(specs):
        X, W, b = si.make_inputs(si.Layer(f"graph_{name}", M, N, K, precision, bias=True))
        inputs[name] = (X, W, b)
    dev = {n: (torch.from_numpy(X).to(dt).cuda(), torch.from_numpy(W).to(dt).cuda(), torch.from_numpy(b).cuda())
           for n, (X, W, b) in inputs.items()}
    x = dev["qkv"][0]
    attn = dev["proj"][0]
    outs = {n: torch.empty((M, N), device="cuda", dtype=dt) for n, N, _, _ in specs}

    def layer():
        tll.forward(x, dev["qkv"][1], dev["qkv"][2], precision=prec, out=outs["qkv"])
        tll.forward(attn, dev["proj"][1], dev["proj"][2], precision=prec, out=outs["proj"])
        tll.forward(x, dev["fc1"][1], dev["fc1"][2], epilogue="gelu", precision=prec, out=outs["fc1"])
        tll.forward(outs["fc1"], dev["fc2"][1], dev["fc2"][2], precision=prec, out=outs["fc2"])

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        layer()  # first calls outside the capture (kernel attributes, device lookups)
        layer()  # and the same call history as the captured calls (adaptive plans)
    stream.synchronize()
    eager = {n: t.clone() for n, t in outs.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer()
    for t in outs.values():
        t.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for n in outs:
        assert torch.equal(outs[n], eager[n]), n
    tll.default_context(0).check()
    # fc1 and fc2 against the oracle (fc2 on the GPU's fc1 output)
    X, W, b = inputs["fc1"]
    tol = oracle.TOL[precision]
    assert oracle.rel_err(outs["fc1"].double().cpu().numpy(), oracle.linear(X, W, b, True)) <= tol
    H = outs["fc1"].float().cpu().numpy()
    _, W2, b2 = inputs["fc2"]
    assert oracle.rel_err(outs["fc2"].double().cpu().numpy(), oracle.linear(H, W2, b2)) <= tol


@pytest.mark.parametrize("K", [4096, 4104, 384, 200])
def test_skinny_bits_independent_of_split(ctx, K):
    """The cluster split only changes who adds which K segments, never the
    shape of the summation tree: every split gives the same bits (so the
    library may choose the split per call without changing results)."""
    X, W, b = si.make_inputs(si.Layer("split_inv", 16, 1024, K, BF16, bias=True))
    for v in range(5):
        outs = [run(X, W, b, BF16, plan=tll.plan_make(ctx.sm_count, tll.KERNEL_SKINNY, v, cl, 16, 1024, K, "bf16"),
                    ctx=ctx) for cl in (1, 2, 4, 8)]
        for o in outs[1:]:
            assert np.array_equal(o, outs[0]), f"variant {v}"
