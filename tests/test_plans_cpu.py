"""The host-side dispatch over a wide grid of shapes (no GPU): every plan
the built-in table returns, and every plan lin_plan_make builds, passes the
same validation lin_forward_plan applies (lin_plan_check), fits the
workspace it was made for, and keeps its grid within the launch limits.
Broken plans (a grid one too large, a split the kernel does not have, too
little workspace) are refused."""
import itertools

import pytest

import transformer_linear_layer_gb300 as tll

SMS = (152, 148, 132)
MS = (1, 2, 3, 4, 5, 8, 9, 15, 16, 17, 31, 64, 100, 127, 128, 129, 200, 255, 256, 257, 1000, 4096, 8192, 40000)
NS = (1, 7, 8, 64, 100, 136, 768, 2304, 3072, 4096, 50257)
KS = (8, 24, 64, 72, 136, 520, 768, 3072, 4096, 4104, 16384)
PRECS = ("fp32", "tf32", "bf16")
WORKSPACES = (0, 1 << 20, 64 << 20)


def _valid_k(K, prec):
    """K rows of X and W must be 16-byte multiples (the ABI's alignment rule)."""
    return (K * (2 if prec == "bf16" else 4)) % 16 == 0


def _grid_ok(p: tll.Plan):
    return 1 <= p.grid_x < 2 ** 31 and 1 <= p.grid_y <= 65535 and 1 <= p.grid_z <= 65535


def test_every_table_plan_passes_validation():
    checked = 0
    for sm, M, N, K, prec, ws in itertools.product(SMS, MS, NS, KS, PRECS, WORKSPACES):
        if not _valid_k(K, prec):
            continue
        for epi in ("none", "gelu"):
            p = tll.plan_query(sm, M, N, K, prec, epi, workspace_bytes=ws)
            rc = tll.plan_check(p, M, N, K, prec, ws)
            assert rc == tll.OK, (sm, M, N, K, prec, epi, ws, p, rc)
            assert p.workspace_bytes <= ws
            assert _grid_ok(p), (sm, M, N, K, prec, p)
            if p.kernel == tll.KERNEL_TC and p.splits == 1 and p.grid_z == 1:
                assert p.grid_x <= sm  # persistent: at most one CTA per SM
            checked += 1
    assert checked > 50000


def test_table_routes():
    """Each precision reaches the families the table is meant to use."""
    seen = {prec: set() for prec in PRECS}
    for M, N, K, prec in itertools.product(MS, NS, KS, PRECS):
        if _valid_k(K, prec):
            seen[prec].add(tll.plan_query(152, M, N, K, prec).kernel)
    assert seen["bf16"] == {tll.KERNEL_GEMV, tll.KERNEL_SKINNY, tll.KERNEL_TC}
    assert seen["tf32"] == {tll.KERNEL_GEMV, tll.KERNEL_TC}
    assert seen["fp32"] == {tll.KERNEL_GEMV, tll.KERNEL_FFMA}


def _family_plans(sm, M, N, K, prec):
    out = []
    menu = []
    if prec == "bf16":
        menu += [(tll.KERNEL_SKINNY, v, s) for v in range(5) for s in (0, 1, 2, 4, 8)]
    if prec in ("bf16", "tf32"):
        menu += [(tll.KERNEL_TC, v, w) for v in range(6) for w in (0, 1, 3, sm)]
        menu += [(tll.KERNEL_TC, v, -c) for v in range(3) for c in (1, 2, 5)]
    if prec == "fp32":
        menu += [(tll.KERNEL_FFMA, v, s) for v in range(4) for s in (0, 1, 2, 3, 7, 12)]
    menu += [(tll.KERNEL_GEMV, 0, c) for c in (0, 3)]
    for kernel, v, s in menu:
        try:
            out.append(tll.plan_make(sm, kernel, v, s, M, N, K, prec))
        except tll.LinError:
            pass
    return out


@pytest.mark.parametrize("prec", PRECS)
def test_every_family_plan_passes_validation(prec):
    made = 0
    for M, N, K in itertools.product((1, 4, 16, 100, 129, 1000, 8192), (7, 136, 768, 3072, 50257),
                                     (24, 136, 768, 3072, 4104)):
        if not _valid_k(K, prec):
            continue
        for p in _family_plans(152, M, N, K, prec):
            rc = tll.plan_check(p, M, N, K, prec, 1 << 62)
            assert rc == tll.OK, (M, N, K, prec, p, rc)
            assert _grid_ok(p)
            made += 1
    assert made > 300


def test_broken_plans_are_refused():
    M, N, K = 1000, 768, 3072
    for prec in PRECS:
        for p in _family_plans(152, M, N, K, prec):
            for field, delta in (("grid_y", 1), ("bn", 8), ("variant", 17)):
                q = tll.Plan.from_buffer_copy(p)
                setattr(q, field, getattr(q, field) + delta)
                rc = tll.plan_check(q, M, N, K, prec, 1 << 62)
                assert rc != tll.OK or (field == "bn" and p.kernel in (tll.KERNEL_FFMA, tll.KERNEL_SKINNY,
                                                                        tll.KERNEL_GEMV)), (field, p)
            if p.workspace_bytes > 0:
                assert tll.plan_check(p, M, N, K, prec, p.workspace_bytes - 1) == tll.ERR_WORKSPACE
    # a kernel for the wrong precision, the wrong shape, or an empty call
    tc = tll.plan_make(152, tll.KERNEL_TC, 0, 0, M, N, K, "bf16")
    assert tll.plan_check(tc, M, N, K, "fp32", 1 << 62) == tll.ERR_UNSUPPORTED
    assert tll.plan_check(tc, M, 2 * N, K, "bf16", 1 << 62) == tll.OK  # persistent CTAs walk any tile count
    assert tll.plan_check(tc, 100, 64, K, "bf16", 1 << 62) == tll.ERR_UNSUPPORTED  # more CTAs than tiles
    ff = tll.plan_make(152, tll.KERNEL_FFMA, 0, 1, M, N, K, "fp32")
    assert tll.plan_check(ff, M, 2 * N, K, "fp32", 1 << 62) == tll.ERR_UNSUPPORTED  # one CTA per tile
    assert tll.plan_check(tc, 0, N, K, "bf16", 1 << 62) == tll.ERR_UNSUPPORTED
    assert tll.plan_check(tll.plan_query(152, 0, N, K, "bf16"), 0, N, K, "bf16", 0) == tll.OK
    assert tll.library().lin_plan_check(None, M, N, K, 2, 0) == tll.ERR_ARG


# ---------------------------------------------------------------- the table's rules


def _cdiv(a, b):
    return -(-a // b)


def test_skinny_cluster_rule():
    """Skinny calls take the 5 x 1 ring (two CTAs per SM) and the largest
    cluster (a power of two, at most 8) that keeps the grid within two CTAs per
    SM and at least two K stages per CTA; the 6 x 1 ring without a split when W
    has more 128-row tiles than SMs."""
    for sm in SMS:
        for M in (2, 8, 16):
            for N in (136, 768, 4096, 16384, 50257):
                for K in (64, 768, 4096):
                    p = tll.plan_query(sm, M, N, K, "bf16")
                    assert p.kernel == tll.KERNEL_SKINNY
                    tiles = _cdiv(N, 128)
                    if tiles > sm:
                        assert p.variant == 1 and p.splits == 1, (sm, M, N, K, p)
                        continue
                    assert p.variant == 4
                    kblocks = _cdiv(K, 64)
                    S = 1
                    while S < 8 and tiles * S * 2 <= 2 * sm and 2 * S <= kblocks:
                        S *= 2
                    assert p.splits == S and p.grid_x == tiles and p.grid_y == S, (sm, M, N, K, p)


def test_ffma_split_rule():
    """FP32: 128x128 tiles (K in steps of 64) when they give a full wave; else
    64x64 tiles split so that the (tile, split) CTAs fill two per SM without a
    second wave, with at least 4 K steps of 32 per split and at least 16 steps
    in all, within the workspace."""
    for sm in SMS:
        for M in (9, 64, 128, 256, 1024, 4096):
            for N in (64, 768, 2304, 3072, 4096):
                for K in (64, 256, 512, 768, 3072):
                    for ws in (0, 64 << 20):
                        p = tll.plan_query(sm, M, N, K, "fp32", workspace_bytes=ws)
                        assert p.kernel == tll.KERNEL_FFMA
                        big = _cdiv(M, 128) * _cdiv(N, 128)
                        assert p.variant == (2 if big >= sm else 1)
                        tm = 128 if p.variant == 2 else 64
                        tiles = _cdiv(M, tm) * _cdiv(N, tm)
                        slots = sm if p.variant == 2 else 2 * sm
                        steps = _cdiv(K, p.bk)
                        assert tiles * p.splits <= max(slots, tiles)
                        assert p.splits == 1 or (steps // p.splits >= 4 and steps >= 16)
                        assert p.workspace_bytes <= ws
                        if ws and 2 * tiles <= slots and steps >= 16:
                            assert p.splits > 1, (sm, M, N, K, p)  # room for two CTAs per tile


def test_tc_k_split_rule():
    """tcgen05 K split: of every tile only when the tiles fill at most half of
    the SMs, with at least 32 K stages per split, at most 16 splits, never for
    the SM pair; a ragged last round is not split by the table (explicit
    plans only); the pair for long K otherwise."""
    for sm in SMS:
        for M in (32, 128, 256, 1024, 8192):
            for N in (256, 768, 3072):
                for K in (768, 2048, 4096, 16384):
                    p = tll.plan_query(sm, M, N, K, "bf16")
                    assert p.kernel == tll.KERNEL_TC
                    pair = p.variant >= 3
                    if p.grid_z > 1:
                        tiles = _cdiv(M, 128) * _cdiv(N, p.bn)
                        assert not pair and p.grid_z <= 16
                        assert tiles * 2 <= sm, (sm, M, N, K, p)
                        assert _cdiv(K, 64) // p.grid_z >= 32
                    if pair:
                        assert _cdiv(K, 64) >= 64
