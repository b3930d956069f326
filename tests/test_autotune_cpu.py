"""The tuner's search and selection logic on the CPU, driven by a fake
context and a synthetic timing backend (no GPU): the paired, same-window
choice, the stopping rule, the pruning, and installing only a real winner.

"Optimizing a GPT-2-class transformer on a GPU" (Act V) records the failure
these tests guard against: measurement was paired but selection compared a
candidate with a stale incumbent number from a warmer window."""
import random

import pytest

import transformer_linear_layer_gb300 as tll
from transformer_linear_layer_gb300 import autotune

SM, WS = 152, 64 << 20


class FakeCtx:
    sm_count, workspace_bytes = SM, WS

    def __init__(self):
        self.overrides = {}

    def plan(self, M, N, K, precision="bf16", epilogue="none"):
        return tll.plan_query(SM, M, N, K, precision, epilogue, WS)

    def set_override(self, M, N, K, precision, epilogue, plan):
        key = (M, N, K, precision, epilogue)
        if plan is None:
            self.overrides.pop(key, None)
        else:
            assert tll.plan_check(plan, M, N, K, precision, WS) == tll.OK
            self.overrides[key] = autotune._plan_key(plan)

    def check(self, stream=None):
        pass


class FakeBench:
    """Seconds per call from a table keyed by plan (None = the incumbent),
    with a 'window' drift: every timing after the first `warm` ones is
    multiplied by `drift`, as if the machine got slower (or faster)."""

    def __init__(self, times, noise=0.0, drift=1.0, warm=0, seed=0, screen_bias=None):
        self.times, self.noise, self.drift, self.warm = times, noise, drift, warm
        self.rng = random.Random(seed)
        self.calls = []
        self.screen_bias = screen_bias or {}
        self.stream = None

    def __call__(self, ctx, M, N, K, precision, epilogue, reps=20):
        return self

    def graph(self, plan):
        return None if plan is None else autotune._plan_key(plan)

    def time(self, g):
        self.calls.append(g)
        t = self.times.get(g, self.times["default"])
        if g in self.screen_bias and self.calls.count(g) == 1:
            t *= self.screen_bias[g]  # a lucky (or unlucky) first timing
        if len(self.calls) > self.warm:
            t *= self.drift
        return t * (1.0 + self.noise * self.rng.uniform(-1, 1))


SHAPE = (128, 768, 768, "fp32", "none")  # FFMA candidates: v0/v1 x splits


def _menu():
    M, N, K, prec, _ = SHAPE
    inc = tll.plan_query(SM, M, N, K, prec, "none", WS)
    return inc, [p for p in autotune.candidates(SM, M, N, K, prec, WS)
                 if autotune._plan_key(p) != autotune._plan_key(inc)]


def test_paired_winner_is_installed():
    inc, cands = _menu()
    best = cands[1]
    times = {"default": 10e-6, None: 8e-6, autotune._plan_key(best): 6e-6}
    ctx, bench = FakeCtx(), FakeBench(times, noise=0.01)
    (rep,) = autotune.autotune(ctx, [SHAPE], bench_factory=bench)
    assert rep["winner"] is not None and autotune._plan_key(autotune._plan_from_dict(rep["winner"])) == \
        autotune._plan_key(best)
    assert abs(rep["winner_ratio"] - 0.75) < 0.03
    assert ctx.overrides[SHAPE] == autotune._plan_key(best)


def test_no_winner_within_margin_installs_nothing():
    inc, cands = _menu()
    times = {"default": 10e-6, None: 8e-6, autotune._plan_key(cands[0]): 7.9e-6}  # 1.3% better: noise
    ctx = FakeCtx()
    (rep,) = autotune.autotune(ctx, [SHAPE], bench_factory=FakeBench(times))
    assert rep["winner"] is None and SHAPE not in ctx.overrides


def test_lucky_screen_timing_does_not_win():
    """A candidate whose single screening timing was lucky (40% low) but which
    is 10% slower in the paired rounds is not chosen."""
    inc, cands = _menu()
    k = autotune._plan_key(cands[0])
    times = {"default": 10e-6, None: 8e-6, k: 8.8e-6}
    ctx = FakeCtx()
    (rep,) = autotune.autotune(ctx, [SHAPE], bench_factory=FakeBench(times, screen_bias={k: 0.6}))
    assert any(p["plan"] == autotune._label(cands[0]) for p in rep["paired"])  # it got paired ...
    assert rep["winner"] is None                                               # ... and lost


def test_selection_is_paired_not_against_a_stale_incumbent():
    """The machine slows down 30% after the incumbent's first timing (a warm
    first window): against that stale number every candidate would look 30%
    slower and nothing would be found; re-timing the incumbent beside each
    candidate finds the real 20% winner."""
    inc, cands = _menu()
    k = autotune._plan_key(cands[2])
    times = {"default": 10e-6, None: 8e-6, k: 6.4e-6}
    bench = FakeBench(times, drift=1.3, warm=1)
    ctx = FakeCtx()
    (rep,) = autotune.autotune(ctx, [SHAPE], bench_factory=bench)
    assert rep["winner"] is not None and abs(rep["winner_ratio"] - 0.8) < 1e-9
    # every candidate timing in the pairs sits between two incumbent timings
    paired = [i for i, g in enumerate(bench.calls) if g == k]
    assert all(bench.calls[i - 1] is None for i in paired[1:])


def test_stopping_rule_skips_search():
    """An incumbent already at its roofline floor is not searched."""
    floor = autotune.roofline_floor_s(*SHAPE[:4])
    bench = FakeBench({"default": 10 * floor, None: floor / 0.98})
    (rep,) = autotune.autotune(FakeCtx(), [SHAPE], bench_factory=bench)
    assert rep["stopped"] and rep["screened"] == [] and bench.calls == [None]


def test_pruning_needs_a_fit_that_knows_the_family():
    """With a residual fit trained on this family, candidates it predicts far
    above the incumbent are not timed; a fresh model times everything."""
    inc, cands = _menu()
    times = {"default": 50e-6, None: 5e-6}
    fresh = FakeBench(times)
    autotune.autotune(FakeCtx(), [SHAPE], bench_factory=fresh)
    assert len(set(g for g in fresh.calls if g is not None)) == len(cands)
    model = autotune.ResidualModel()
    for _ in range(3):  # teach it that this family runs 10x its prior
        autotune.autotune(FakeCtx(), [SHAPE], bench_factory=FakeBench(times), model=model)
    assert model.knows(autotune.features(SM, *SHAPE[:4], cands[0]))
    taught = FakeBench(times)
    (rep,) = autotune.autotune(FakeCtx(), [SHAPE], bench_factory=taught, model=model)
    assert rep["pruned"] and len(set(g for g in taught.calls if g is not None)) < len(cands)


def test_unknown_family_is_not_pruned():
    model = autotune.ResidualModel()
    f_known = {"fill": 0.5, "tile_fill": 1.0, "split": 1, "family": "ffma", "stream_k": False}
    for _ in range(30):
        model.add(f_known, 1e-5, 1e-6)
    model.fit()
    assert model.trusted and model.knows(f_known)
    assert not model.knows(dict(f_known, family="gemv"))
