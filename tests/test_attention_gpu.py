"""GPU parity of the fused attention forward (lin_attention_forward) against
the oracle's attention (float64, the two-pass definition).

Tolerance, from the kernel's arithmetic: scores are fp32 sums of exact bf16
products, the probabilities p_ij are rounded to bf16 (round to nearest, 8
significant bits: relative error at most 2^-8) before their product with v,
the row sum l keeps them in fp32, and the output is rounded to bf16 (2^-8
relative). So per output element

    |out - ref| <= 2^-8 (sum_j p_ij |v_j[d]|) + 2^-8 |ref|  (+ fp32 rounding),

and the test allows 5% over that plus 1e-5 for the fp32 sums:
1.05 * 2^-8 (A + |ref|) + 1e-5 with A = sum_j p_ij |v_j[d]| computed here in
float64. lse: fp32 scores, fp32 sums and the hardware log2, within
1e-4 (1 + |lse|).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    return tll.default_context(0)


def weighted_abs(qkv, B, T, H, D, causal, scale):
    """A[b*T + i][h*D + d] = sum_j p_ij |v_j[d]| in float64 (tolerance only)."""
    C = H * D
    x = qkv.astype(np.float64).reshape(B, T, 3, H, D)
    q, k, v = x[:, :, 0], x[:, :, 1], x[:, :, 2]
    s = np.einsum("bihd,bjhd->bhij", q, k) * scale
    if causal:
        s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    s -= s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    a = np.einsum("bhij,bjhd->bihd", p, np.abs(v))
    return a.reshape(B * T, C)


def run_attention(ctx, att: si.Attention, scale=None, with_lse=True):
    qkv = si.make_qkv(att)
    dq = torch.from_numpy(qkv).to(torch.bfloat16).cuda()
    out, lse = tll.attention_forward(dq, att.B, att.T, att.H, causal=att.causal, scale=scale, with_lse=True,
                                     ctx=ctx)
    ctx.check()
    return qkv, out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(ctx, att: si.Attention, scale=None):
    qkv, out, lse = run_attention(ctx, att, scale)
    sc = 1.0 / np.sqrt(att.D) if scale is None else scale
    ref, ref_lse = oracle.attention(qkv, att.B, att.T, att.H, att.D, causal=att.causal, scale=sc, with_lse=True)
    A = weighted_abs(qkv, att.B, att.T, att.H, att.D, att.causal, sc)
    bound = 1.05 * 2.0 ** -8 * (A + np.abs(ref)) + 1e-5
    err = np.abs(out - ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (att, worst, out[worst], ref[worst], bound[worst])
    lerr = np.abs(lse - ref_lse)
    assert np.all(lerr <= 1e-4 * (1 + np.abs(ref_lse))), (att, float(lerr.max()))
    return float(np.max(err / bound))


CASES = [
    # (B, T, H, causal): one block, several key blocks, ragged T, T below one block, one token
    (1, 128, 1, True), (1, 128, 1, False),
    (2, 256, 3, True), (2, 256, 3, False),
    (2, 200, 2, True), (2, 200, 2, False),
    (3, 384, 2, True), (1, 520, 1, False),
    (2, 5, 2, True), (3, 1, 2, False), (4, 77, 3, True),
]


@pytest.mark.parametrize("B,T,H,causal", CASES)
def test_attention_matches_oracle(ctx, B, T, H, causal):
    check(ctx, si.Attention(f"attn_{B}x{T}x{H}", B, T, H, 64, causal=causal, seed=B * 1000 + T + H))


@pytest.mark.parametrize("scale", [1.0, 0.01])
def test_attention_peaked_and_flat_softmax(ctx, scale):
    """scale 1: scores of spread 8, so the running max changes from block to
    block and most rows are dominated by a few keys; 0.01: nearly uniform."""
    check(ctx, si.Attention("attn_scale", 2, 384, 2, 64, causal=True, seed=7), scale=scale)
    check(ctx, si.Attention("attn_scale_full", 2, 300, 2, 64, causal=False, seed=8), scale=scale)


def test_attention_gpt2_batched_shape(ctx):
    """GPT-2 small's attention at 64 sequences x 128 tokens x 12 heads, the
    benchmark's launch, every output element against the oracle."""
    check(ctx, si.GPT2_ATTN_B64)


def test_attention_is_repeatable_and_leaves_neighbours(ctx):
    att = si.Attention("attn_rep", 3, 200, 4, 64, causal=True, seed=3)
    dq = torch.from_numpy(si.make_qkv(att)).to(torch.bfloat16).cuda()
    C = att.C
    big = torch.full((att.B * att.T + 2, C), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[1:-1]
    tll.attention_forward(dq, att.B, att.T, att.H, out=out, ctx=ctx)
    first = out.clone()
    tll.attention_forward(dq, att.B, att.T, att.H, out=out, ctx=ctx)
    ctx.check()
    assert torch.equal(first, out)
    assert torch.all(big[0] == 7.0) and torch.all(big[-1] == 7.0)


def test_attention_argument_errors(ctx):
    lib = tll.library()
    dq = torch.zeros((256, 3 * 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((256, 128), dtype=torch.bfloat16, device="cuda")
    h = ctx._h
    ok = lib.lin_attention_forward(h, 2, 128, 2, 64, dq.data_ptr(), out.data_ptr(), None, 1, 0.0, None)
    assert ok == tll.OK
    assert lib.lin_attention_forward(h, 2, 128, 2, 32, dq.data_ptr(), out.data_ptr(), None, 1, 0.0, None) \
        == tll.ERR_UNSUPPORTED
    assert lib.lin_attention_forward(h, 2, 128, 2, 64, dq.data_ptr(), out.data_ptr(), None, 2, 0.0, None) \
        == tll.ERR_ARG
    assert lib.lin_attention_forward(h, 2, 128, 2, 64, dq.data_ptr(), out.data_ptr(), None, 1, -1.0, None) \
        == tll.ERR_ARG
    assert lib.lin_attention_forward(h, 2, 128, 2, 64, dq.data_ptr(), dq.data_ptr(), None, 1, 0.0, None) \
        == tll.ERR_ARG  # out overlaps qkv
    wide = torch.zeros((256 + 8, 3 * 128), dtype=torch.bfloat16, device="cuda")  # room for a 2-byte shift
    assert lib.lin_attention_forward(h, 2, 128, 2, 64, wide.data_ptr() + 2, out.data_ptr(), None, 1, 0.0, None) \
        == tll.ERR_ALIGN
    assert lib.lin_attention_forward(h, 2, 128, 2, 64, None, out.data_ptr(), None, 1, 0.0, None) == tll.ERR_ARG
    # nothing to do
    assert lib.lin_attention_forward(h, 0, 128, 2, 64, None, None, None, 1, 0.0, None) == tll.OK
    assert lib.lin_attention_forward(h, 2, 0, 2, 64, None, None, None, 1, 0.0, None) == tll.OK
    ctx.check()
