"""Measured dispatch: time candidate plans for given call signatures and install
the winners in a context.

"Optimizing a GPT-2-class transformer on a GPU" (Act II) ends in a routing
table, each shape sent to its measured winner, and its Act V turns the search
for that table into a loop with four ports, which this module fills for the
library's own kernels:

- what may be proposed: only the resource knees (tile widths, SM pairs, K
  splits, stream-K, the skinny ring and cluster sizes, the FFMA split
  counts, the GEMV), each a plan the library has checked for the shape;
- how cost is predicted: a roofline with penalties (waves that leave SMs
  idle, padded tile area, the split's partial sums through HBM) as the
  prior, and a least-squares regression on the same physical features that
  learns only the prior's error (the residual), refit after every shape;
  its coefficients say which penalty the prior over- or underprices;
- which experiment runs next: candidates the corrected model puts far above
  the incumbent are pruned before any timing, unless their family is one
  the fit has barely seen (where it is uncertain); the rest are timed once;
- how a result is scored: as efficiency, the physical floor (the layer's
  own roofline) over the time, with a stopping rule (an incumbent already
  at ``stop`` of its floor is not searched), and the choice is paired:
  the best timed candidates alternate with the incumbent in one window,
  ``rounds`` times, and one wins only when its median time ratio is below
  ``1 - margin``.

The incumbent is timed through ``lin_forward`` itself (the built-in table,
with its adaptive choices), a candidate through ``lin_forward_plan`` (which an
installed override also uses): both back to back on one stream with the
context's early-start level (LIN_OPT_EARLY_START), with the weight rotated
over enough copies to exceed the L2, so that each call reads its weight from
HBM as a layer of a model does. Winners are found for the context as it is
configured: tune with the early-start level the caller will run with.
"""
from __future__ import annotations

import json
import math
import statistics

from . import (KERNEL_FFMA, KERNEL_GEMV, KERNEL_NAMES, KERNEL_SKINNY, KERNEL_TC, Context, LinError, Plan,
               PREC_BF16, PREC_FP32, PREC_TF32, _epi, _prec, plan_make)

_PLAN_FIELDS = ("kernel", "variant", "bm", "bn", "bk", "splits", "stages", "grid_x", "grid_y", "grid_z", "threads",
                "workspace_bytes")


def _plan_key(p: Plan):
    return tuple(getattr(p, f) for f in _PLAN_FIELDS)


def _plan_from_dict(d) -> Plan:
    p = Plan()
    for f in _PLAN_FIELDS:
        setattr(p, f, int(d[f]))
    return p


def candidates(sm_count: int, M: int, N: int, K: int, precision, workspace_bytes: int):
    """The plans that can run this shape (host only): a deduplicated list."""
    prec = _prec(precision)
    name = {PREC_FP32: "fp32", PREC_TF32: "tf32", PREC_BF16: "bf16"}[prec]
    out, seen = [], set()

    def add(kernel, variant, splits):
        try:
            p = plan_make(sm_count, kernel, variant, splits, M, N, K, name)
        except LinError:
            return
        if p.workspace_bytes > workspace_bytes:
            return
        k = _plan_key(p)
        if k not in seen:
            seen.add(k)
            out.append(p)

    if prec == PREC_BF16 and M <= 16:
        for v in range(5):  # the skinny kernel's ring variants
            for s in (1, 2, 4, 8):
                add(KERNEL_SKINNY, v, s)
    if prec in (PREC_BF16, PREC_TF32):
        for v in range(6):
            add(KERNEL_TC, v, 0)
        for v in range(3):
            add(KERNEL_TC, v, -1)  # stream-K
    if prec == PREC_FP32:
        for v in range(4):  # FFMA tile variants (lin_plan variant ids)
            for s in (1, 2, 3, 4, 6, 8, 12):
                add(KERNEL_FFMA, v, s)
    if M <= 8:
        add(KERNEL_GEMV, 0, 0)
    return out


def roofline_floor_s(M, N, K, precision, peaks=None) -> float:
    """max(bytes / HBM, FLOPs / peak) for the layer (X, W, Y once each)."""
    prec = _prec(precision)
    peaks = peaks or {"hbm_gbs": 6783.1, "bf16_tflops": 1891.6}
    esz = 2 if prec == PREC_BF16 else 4
    byts = (M * K + N * K + M * N) * esz
    if prec == PREC_BF16:
        peak = peaks["bf16_tflops"] * 1e12
    elif prec == PREC_TF32:
        peak = peaks["bf16_tflops"] * 1e12 * (1.1 / 2.25)
    else:
        peak = 152 * 128 * 2 * 2.07e9
    return max(byts / (peaks["hbm_gbs"] * 1e9), 2.0 * M * N * K / peak)


_FFMA_TFLOPS = 152 * 128 * 2 * 2.07e-3  # SMs x fp32 lanes x 2 FLOPs x GHz -> TF/s


def features(sm: int, M: int, N: int, K: int, precision, p: Plan) -> dict:
    """Physical features of a plan on a shape: ``fill`` (work units over the
    slots their waves occupy), ``tile_fill`` (output area over padded tile
    area), ``split`` (K split factor) and the family."""
    prec = _prec(precision)
    split = 1
    if p.kernel == KERNEL_TC:
        pair = p.variant >= 3
        bm = 256 if pair else 128
        units = -(-M // bm) * -(-N // p.bn) * max(p.grid_z, 1)
        slots = min(sm // 2 if pair else sm, max(p.grid_x // (2 if pair else 1), 1) * max(p.grid_z, 1))
        slots = max(slots, 1)
        split = max(p.grid_z, 1)
        mpad, npad = -(-M // bm) * bm, -(-N // p.bn) * p.bn
        fam = "tc_pair" if pair else "tc"
    elif p.kernel == KERNEL_SKINNY:
        per_sm = 2 if p.stages * (p.bk // 64) * 16 <= 96 else 1  # ring KB: 192 -> one CTA per SM
        units, slots = p.grid_x * p.grid_y, sm * per_sm
        split = p.grid_y
        mpad, npad = 16, -(-N // 128) * 128
        fam = "skinny"
    elif p.kernel == KERNEL_FFMA:
        units, slots = p.grid_x * p.grid_y * p.grid_z, sm * (2 if p.variant in (1, 3) else 1)
        split = p.grid_z
        mpad, npad = -(-M // p.bm) * p.bm, -(-N // p.bn) * p.bn
        fam = "ffma"
    else:  # GEMV: the CTAs walk the rows of W
        units = slots = max(p.grid_x, 1)
        mpad, npad = max(p.bm, 1), N
        fam = "gemv"
    waves = -(-units // slots)
    return {"fill": units / (waves * slots), "tile_fill": (M * N) / max(mpad * npad, 1), "split": split,
            "family": fam, "stream_k": p.kernel == KERNEL_TC and p.splits == 2}


def predict_prior_s(M, N, K, precision, f: dict, peaks=None) -> float:
    """Roofline with penalties: compute at the family's peak scaled by the wave
    and tile fill, bytes at HBM speed plus the split's fp32 partials (written
    and read once per extra split; the skinny kernel adds its partials on
    chip)."""
    prec = _prec(precision)
    peaks = peaks or {"hbm_gbs": 6783.1, "bf16_tflops": 1891.6}
    esz = 2 if prec == PREC_BF16 else 4
    byts = (M * K + N * K + M * N) * esz
    if f["family"] != "skinny":
        byts += (f["split"] - 1) * M * N * 4 * 2
    if f["family"] in ("ffma", "gemv"):
        peak = _FFMA_TFLOPS * 1e12
    elif prec == PREC_TF32:
        peak = peaks["bf16_tflops"] * 1e12 * (1.1 / 2.25)
    else:
        peak = peaks["bf16_tflops"] * 1e12
    return max(byts / (peaks["hbm_gbs"] * 1e9), 2.0 * M * N * K / (peak * f["fill"] * f["tile_fill"]))


# log(1/fill) and log(1/tile_fill) are the prior's own penalties in log form:
# a coefficient of -1 cancels one, 0 keeps it as priced.
_FEATURE_NAMES = ("bias", "log_idle_waves", "log_tile_padding", "log2_split", "stream_k", "sm_pair", "skinny",
                  "ffma", "gemv")


def _phi(f: dict):
    return [1.0, math.log(1.0 / f["fill"]), math.log(1.0 / f["tile_fill"]), math.log2(max(f["split"], 1)),
            1.0 if f["stream_k"] else 0.0, 1.0 if f["family"] == "tc_pair" else 0.0,
            1.0 if f["family"] == "skinny" else 0.0, 1.0 if f["family"] == "ffma" else 0.0,
            1.0 if f["family"] == "gemv" else 0.0]


class ResidualModel:
    """log(measured / prior) = phi . beta by ridge least squares (the prior's
    error as a function of its own penalty features)."""

    def __init__(self, ridge: float = 1e-2):
        self.rows, self.ys, self.ridge = [], [], ridge
        self.beta = [0.0] * len(_FEATURE_NAMES)
        self.per_family = {}
        # What the current beta was fitted on: pruning trusts the fit, not
        # samples added since (within a search the fit runs after screening).
        self.n_fit, self.fam_fit = 0, {}

    def add(self, f: dict, measured_s: float, prior_s: float):
        self.rows.append(_phi(f))
        self.ys.append(math.log(measured_s / prior_s))
        self.per_family[f["family"]] = self.per_family.get(f["family"], 0) + 1

    def knows(self, f: dict, min_samples: int = 3) -> bool:
        """The fit has seen this plan's family often enough to prune with it;
        a family it has not seen is exactly where it is uncertain, so such
        candidates are timed, not pruned."""
        return self.trusted and self.fam_fit.get(f["family"], 0) >= min_samples

    @property
    def trusted(self) -> bool:
        """The fit was made on enough samples to prune with (two per feature)."""
        return self.n_fit >= 2 * len(_FEATURE_NAMES)

    def fit(self):
        import numpy as np

        if len(self.ys) < 2:
            return
        A = np.asarray(self.rows)
        y = np.asarray(self.ys)
        reg = self.ridge * np.eye(A.shape[1])
        reg[0, 0] = 0.0  # the intercept is not shrunk
        self.beta = list(np.linalg.solve(A.T @ A + reg, A.T @ y))
        self.n_fit, self.fam_fit = len(self.ys), dict(self.per_family)

    def predict_s(self, f: dict, prior_s: float) -> float:
        return prior_s * math.exp(sum(b * x for b, x in zip(self.beta, _phi(f))))

    def report(self) -> list:
        """One entry per feature: its coefficient and whether the prior
        overprices (negative: faster than the prior says as the feature
        grows) or underprices it."""
        return [{"feature": n, "coef": round(float(b), 4),
                 "prior": "as priced" if abs(b) < 0.02 else ("OVERprices" if b < 0 else "UNDERprices")}
                for n, b in zip(_FEATURE_NAMES, self.beta)]


class _Bench:
    """Back-to-back lin_forward_plan calls of one shape, timed as CUDA graphs."""

    L2_BYTES = 129 << 20

    def __init__(self, ctx: Context, M, N, K, precision, epilogue, reps=20):
        import torch

        self.torch = torch
        self.ctx, self.M, self.N, self.K = ctx, M, N, K
        self.prec, self.epi = _prec(precision), _epi(epilogue)
        dt = torch.bfloat16 if self.prec == PREC_BF16 else torch.float32
        dev = torch.device("cuda", ctx.device)
        g = torch.Generator(device=dev).manual_seed(0)
        w_bytes = N * K * (2 if self.prec == PREC_BF16 else 4)
        copies = max(2, min(64, math.ceil(2 * self.L2_BYTES / max(w_bytes, 1))))
        self.x = torch.randn((M, K), device=dev, generator=g).to(dt)
        self.ws = [(torch.randn((N, K), device=dev, generator=g) * 0.02).to(dt) for _ in range(copies)]
        self.bias = torch.randn((N,), device=dev, generator=g) * 0.02
        self.y = torch.empty((M, N), device=dev, dtype=dt)
        self.stream = torch.cuda.Stream(dev)
        self.reps = max(reps, copies)

    def graph(self, plan: Plan | None):
        """A graph of ``reps`` calls; ``plan`` None = through ``lin_forward``."""
        torch = self.torch
        s = self.stream.cuda_stream

        def step(i):
            args = (self.M, self.N, self.K, self.x.data_ptr(), self.ws[i % len(self.ws)].data_ptr(),
                    self.bias.data_ptr(), self.y.data_ptr(), self.epi, self.prec, s)
            rc = self.ctx.forward_ptr(*args) if plan is None else self.ctx.forward_plan_ptr(plan, *args)
            if rc != 0:
                raise LinError(rc, "lin_forward_plan")

        with torch.cuda.stream(self.stream):
            for i in range(3):
                step(i)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(self.reps):
                    step(i)
        self.stream.synchronize()
        return g

    def time(self, g) -> float:
        torch = self.torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            g.replay()
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
        self.stream.synchronize()
        return e0.elapsed_time(e1) / 1e3 / self.reps


def autotune(ctx: Context, shapes, rounds: int = 5, reps: int = 20, prune: float = 2.0, slack: float = 0.15,
             pair_top: int = 4, margin: float = 0.03, stop: float = 0.97, install: bool = True,
             model: ResidualModel | None = None, bench_factory=None):
    """Tune each (M, N, K, precision, epilogue) in ``shapes``; returns one
    report dict per shape (the incumbent, the efficiencies, the screened and
    paired candidates and the winner, None when the built-in plan stays) and,
    with ``install``, installs the winners (an old override for a tuned shape
    is removed first). ``model`` (refit after each shape) carries the learnt
    residual from shape to shape and across calls. ``bench_factory(ctx, M, N,
    K, precision, epilogue, reps)`` makes the timing backend (default: CUDA
    graphs of back-to-back calls on the context's device): an object with
    ``graph(plan or None)``, ``time(graph) -> seconds per call`` and ``stream``."""
    model = model if model is not None else ResidualModel()
    bench_factory = bench_factory or _Bench
    reports = []
    for (M, N, K, precision, epilogue) in shapes:
        ctx.set_override(M, N, K, precision, epilogue, None)  # time the built-in table, not an old winner
        incumbent = ctx.plan(M, N, K, precision, epilogue)
        bench = bench_factory(ctx, M, N, K, precision, epilogue, reps=reps)
        g_inc = bench.graph(None)
        t_inc = bench.time(g_inc)
        floor = roofline_floor_s(M, N, K, precision)
        rep = {"shape": [M, N, K], "precision": precision, "epilogue": epilogue,
               "roofline_floor_us": floor * 1e6, "incumbent_us": t_inc * 1e6, "incumbent": incumbent.as_dict(),
               "efficiency": floor / t_inc, "winner": None, "winner_ratio": 1.0, "pruned": [], "screened": [],
               "paired": [], "stopped": floor / t_inc >= stop}
        reports.append(rep)
        if rep["stopped"]:  # at the floor already: nothing to find
            continue
        cands = [p for p in candidates(ctx.sm_count, M, N, K, precision, ctx.workspace_bytes)
                 if _plan_key(p) != _plan_key(incumbent)]
        graphs, screen = {}, []
        for p in cands:
            f = features(ctx.sm_count, M, N, K, precision, p)
            prior = predict_prior_s(M, N, K, precision, f)
            # analytic pruning before the stopwatch, where the residual has data behind it
            if model.knows(f) and model.predict_s(f, prior) > prune * t_inc:
                rep["pruned"].append(_label(p))
                continue
            try:
                graphs[_plan_key(p)] = bench.graph(p)
            except LinError:
                continue
            t = bench.time(graphs[_plan_key(p)])
            screen.append((t, p))
            model.add(f, t, prior)
            rep["screened"].append({"plan": _label(p), "us": t * 1e6,
                                    "predicted_us": model.predict_s(f, prior) * 1e6})
        ctx.check(bench.stream)
        model.fit()
        # paired, same-window selection: the best few timed candidates against the incumbent
        screen.sort(key=lambda tp: tp[0])
        paired = []
        for t, p in screen[:pair_top]:
            if t > (1.0 + slack) * t_inc:
                break
            g_c = graphs[_plan_key(p)]
            ratios = []
            for _ in range(rounds):
                a = bench.time(g_inc)
                b = bench.time(g_c)
                ratios.append(b / a)
            paired.append((statistics.median(ratios), p))
        ctx.check(bench.stream)
        winner, best = None, 1.0
        for r, p in paired:
            if r < 1.0 - margin and r < best:
                winner, best = p, r
        if install and winner is not None:
            ctx.set_override(M, N, K, precision, epilogue, winner)
        rep["paired"] = [{"plan": _label(p), "median_ratio": r} for r, p in paired]
        if winner is not None:
            rep["winner"], rep["winner_ratio"] = winner.as_dict(), best
            rep["efficiency_tuned"] = floor / (t_inc * best)
        del graphs, g_inc, bench
    for r in reports:
        r["residual_model"] = model.report()
    return reports


def _label(p: Plan) -> str:
    return f"{KERNEL_NAMES.get(p.kernel, '?')} v{p.variant} bn{p.bn} s{p.splits} grid {p.grid_x}x{p.grid_y}x{p.grid_z}"


def save(reports, path: str):
    """Write the winners (one entry per call signature that has one) as JSON."""
    table = [{"shape": r["shape"], "precision": r["precision"], "epilogue": r["epilogue"],
              "plan": {f: r["winner"][f] for f in _PLAN_FIELDS}} for r in reports if r["winner"] is not None]
    with open(path, "w") as f:
        json.dump(table, f, indent=1)


def load(ctx: Context, path: str) -> int:
    """Install the winners of a saved table; returns how many were installed
    (entries that do not fit this context are skipped)."""
    with open(path) as f:
        table = json.load(f)
    n = 0
    for e in table:
        M, N, K = e["shape"]
        try:
            ctx.set_override(M, N, K, e["precision"], e["epilogue"], _plan_from_dict(e["plan"]))
            n += 1
        except LinError:
            pass
    return n


def main(argv=None):
    """``python -m transformer_linear_layer_gb300.autotune M,N,K,precision,epilogue ... [--out plans.json]``:
    tune the given call signatures on device 0 and print one report line each."""
    import argparse

    ap = argparse.ArgumentParser(description=main.__doc__)
    ap.add_argument("shapes", nargs="+", help="M,N,K,precision,epilogue (precision fp32|tf32|bf16, epilogue none|gelu)")
    ap.add_argument("--out", default=None, help="write the winners as JSON (for load())")
    ap.add_argument("--rounds", type=int, default=5)
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args(argv)
    shapes = []
    for s in a.shapes:
        M, N, K, prec, epi = s.split(",")
        shapes.append((int(M), int(N), int(K), prec, epi))
    ctx = Context(0)
    reports = autotune(ctx, shapes, rounds=a.rounds, reps=a.reps)
    for r in reports:
        print(json.dumps({"shape": r["shape"], "precision": r["precision"], "epilogue": r["epilogue"],
                          "roofline_floor_us": round(r["roofline_floor_us"], 2),
                          "incumbent_us": round(r["incumbent_us"], 2),
                          "efficiency": round(r["efficiency"], 3), "stopped": r["stopped"],
                          "incumbent": _label(_plan_from_dict(r["incumbent"])),
                          "winner": None if r["winner"] is None else _label(_plan_from_dict(r["winner"])),
                          "winner_ratio": round(r["winner_ratio"], 4), "pruned": len(r["pruned"]),
                          "screened": [(x["plan"], round(x["us"], 2), round(x["predicted_us"], 2))
                                       for x in r["screened"]],
                          "paired": [(x["plan"], round(x["median_ratio"], 4)) for x in r["paired"]]}))
    if reports:
        print(json.dumps({"residual_model": reports[-1]["residual_model"]}))
    if a.out:
        save(reports, a.out)


if __name__ == "__main__":
    main()
