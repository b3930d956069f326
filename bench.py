"""Benchmark of the GB300 linear layer (one JSON line on stdout).

Default workload: the skinny linear layer, M = 16 vectors against a
4096 x 4096 bf16 weight stored out x in, fp32 accumulate, bf16 output, fp32
bias ("One multiply, one RTX 5090, eight kernels", "The multiply"). A step is
one call of the layer through the C ABI (dispatch, split-K stream of W,
fixed-order reduction, epilogue). Metric: achieved HBM GB/s over the
algorithmic bytes (X + W + Y + bias once each) with W cold: each step reads
one of R identical copies of W (R x 32 MiB > 4 x L2), and the L2 is flushed
by a read of a buffer twice its size before every timed region, so no step
finds its W in L2 (the page's section "Where the time goes" keeps its weights
cold the same way, cycling through copies of them).

Three ways of calling the layer back to back are timed, each over exactly
--steps calls replayed from warm CUDA graphs:
  back_to_back  independent calls (same X, rotating W), the early start at
                level 2: a call may launch and read its inputs before its
                predecessor finishes (the JSON line's `value`);
  isolated_call the library default (no early start): every call waits for
                the previous kernel to finish before it reads anything;
  chained_call  X of call i+1 is Y of call i (a stack of layers), the early
                start at level 1: W streams before the wait, X after it.
Each also reports its steady state over a longer run and the difference (the
pipeline fill and drain that a short run pays once).

`per_config` times every configuration of the benchmark list in the same run
(fp32 256^3, the M = 16 layer, 4096^3 FFMA and TF32, GPT-2 seq-128 fp32 and
batched bf16 layers, the LM head) as isolated and back-to-back calls, each
with its full-output error against the CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --all] [--no-per-config]

--impl reference times the CPU oracle (the plain double-accumulating triple
loop) on the host cores on the same workload. Under torchrun (N > 1) each
rank runs an independent replica (the layer has no cross-GPU exchange);
value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = "GEMM TFLOP/s (GB/s for M=16) per shape and % of GB300 roofline, cold W"
PREC_NAME = {si.PREC_FP32: "fp32", si.PREC_TF32: "tf32", si.PREC_BF16: "bf16"}
WORKLOADS = {w.name: w for w in si.ALL_WORKLOADS}
DEFAULT_WORKLOAD = si.SKINNY_16x4096.name
# The benchmark's configurations, in the order the line lists them.
PER_CONFIG = ((si.SQUARE_256_FP32, si.SKINNY_16x4096, si.SQUARE_4096_FP32, si.SQUARE_4096_TF32) +
              si.GPT2_M128_FP32 + si.GPT2_M8192_BF16)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MAX_GRAPH = 2048  # calls per captured graph


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------- peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def is_hbm_bound(layer) -> bool:
    """The bound of a layer: bytes at the copy peak against FLOPs at the
    tensor peak (the fp32 path is always FFMA-bound at the shapes here)."""
    if layer.precision == si.PREC_FP32:
        return False
    return layer.algorithmic_bytes() / 6.8e12 >= layer.flops / 1.9e15


def roofline_for(layer, seconds_per_launch: float, peaks, peaks_src, traffic, ffma=None):
    """The bound that applies to this layer and the achieved fraction of it.
    `ffma`: the FFMA peak measured in this run ({"tflops": ...}), else the
    nominal unit count x clock."""
    flops = layer.flops
    byts = layer.algorithmic_bytes()
    if is_hbm_bound(layer):
        ach = byts / seconds_per_launch / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"hbm copy, {peaks_src}", "algorithmic_bytes_per_launch": byts}
    if layer.precision == si.PREC_BF16:
        tens, note = peaks["bf16_tflops"] * 1e12, f"bf16 dense burst, {peaks_src}"
    elif layer.precision == si.PREC_TF32:
        tens, note = peaks["bf16_tflops"] * 1e12 * (1.1 / 2.25), f"tf32 = bf16 burst {peaks_src} x 1.1/2.25 nominal"
    elif ffma:
        tens, note = ffma["tflops"] * 1e12, "fp32 FFMA, measured in this run (lin_probe_ffma)"
    else:
        tens = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6
        note = "fp32 FFMA nominal = 152 SMs x 128 lanes x 2 x sm_max_mhz"
    ach = flops / seconds_per_launch / 1e12
    bound = "alu" if layer.precision == si.PREC_FP32 else "tensor"
    return {"bound": bound, "achieved": round(ach, 2), "peak": round(tens / 1e12, 1), "unit": "TFLOP/s",
            "frac": round(ach * 1e12 / tens, 4), "traffic": traffic, "peak_source": note,
            "algorithmic_flops_per_launch": flops}


def traffic_from_profile(kernel_file: str, workload: str, kernel: str | None = None):
    """dram bytes per launch from the committed ncu summary of this kernel and
    workload (profiles/<kernel>_<workload>.md; the kernel name defaults to the
    file's stem + "_kernel"), or None when absent or when the kernel source has
    changed since the capture."""
    kernel = kernel or kernel_file.replace(".cu", "_kernel")
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "transformer_linear_layer_gb300", "csrc", kernel_file)
    try:
        text = open(prof).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != digest:
        return None
    return float(m.group(1))


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        self.fh = os.fdopen(fd, "w")
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-lms", "100", "-i", str(device_index)], stdout=self.fh,
                                     stderr=subprocess.DEVNULL)

    def stop(self):
        if not self.proc:
            return {"error": "nvidia-smi not available"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"error": "no samples"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        smax = [num(r[3]) for r in rows if num(r[3]) is not None]
        pw = [num(r[4]) for r in rows if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [v for v in sm if smax and v >= 0.5 * max(smax)] or sm
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# -------------------------------------------------------------- multi-rank

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def aggregate(local_seconds: float, local_units: float, world: int, device=None):
    """Slowest rank's time and all ranks' units (replicas: no data exchange)."""
    if world == 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_seconds, local_units], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1])


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ timing

class CallTimer:
    """Times exactly n back-to-back calls of `step(i)` (call i) on `stream`.

    The calls are captured in CUDA graphs whose length is a multiple of
    `period` (the W copies rotate with that period, so consecutive replays
    continue the rotation), replayed twice before any timing (a graph's first
    replay pays its upload), and the L2 is flushed by reading a buffer twice
    its size right before the timed region (reads leave no dirty lines for
    the timed calls to write back). The region is bracketed by CUDA events
    on `stream`, with a barrier and a device synchronisation before the
    flush and after the end event."""

    def __init__(self, torch, stream, step, period, flush_buf, world=1):
        self.torch, self.stream, self.step, self.period, self.flush_buf = torch, stream, step, period, flush_buf
        self.world = world
        self.graphs = {}
        self._sink = torch.empty((), dtype=flush_buf.dtype, device=flush_buf.device)

    def _capture(self, n):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(n):
                self.step(i)
        return g

    def _plan(self, n):
        if n not in self.graphs:
            G = max(self.period, (MAX_GRAPH // self.period) * self.period)
            if n <= G:
                parts = [(self._capture(n), 1)]
            else:
                parts = [(self._capture(G), n // G)]
                if n % G:
                    parts.append((self._capture(n % G), 1))
            with self.torch.cuda.stream(self.stream):
                for g, _ in parts:
                    g.replay()
                    g.replay()
            self.stream.synchronize()
            self.graphs[n] = parts
        return self.graphs[n]

    def flush(self):
        with self.torch.cuda.stream(self.stream):
            self.torch.sum(self.flush_buf, dim=0, out=self._sink)

    def measure(self, n) -> float:
        """Seconds for exactly n calls. After the barrier and device
        synchronisation, the L2 flush and a ~0.2 ms spin of the GPU (no memory
        traffic) are enqueued directly before the start event: meanwhile the
        host enqueues the graphs, so the timed region holds the n calls and not
        the host's graph-launch latency, and the calls still find the L2
        cold."""
        torch = self.torch
        parts = self._plan(n)
        self.stream.synchronize()
        barrier(self.world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        self.flush()
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(400_000)  # clock cycles
            e0.record(self.stream)
            for g, reps in parts:
                for _ in range(reps):
                    g.replay()
            e1.record(self.stream)
        self.stream.synchronize()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    def soak(self, seconds):
        """Replay the largest prepared graph for about `seconds` (clocks settle)."""
        parts = max(self.graphs.values(), key=lambda p: p[0][1])
        until = time.perf_counter() + seconds
        with self.torch.cuda.stream(self.stream):
            while time.perf_counter() < until:
                parts[0][0].replay()
                self.stream.synchronize()


def steady_calls(seconds_per_call_guess: float, steps: int, budget_s=0.05, cap=20000) -> int:
    """Calls in the long run that gives a mode's steady state: >= steps, about
    budget_s of work, at most cap."""
    n = int(budget_s / max(seconds_per_call_guess, 1e-7))
    return max(steps, min(cap, n))


def measure_ffma_peak(torch, ctx, dev, stream):
    """The fp32 FMA pipe's throughput from lin_probe_ffma (CUDA events, after
    a warm-up launch): the FFMA kernels' roofline in this run."""
    out = torch.zeros(1, device=dev)
    iters = 4096
    with torch.cuda.stream(stream):
        ctx.probe_ffma_ptr(iters, out.data_ptr(), stream.cuda_stream)
    stream.synchronize()
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            flops = ctx.probe_ffma_ptr(iters, out.data_ptr(), stream.cuda_stream)
            e1.record(stream)
        stream.synchronize()
        s = e0.elapsed_time(e1) / 1e3
        best = s if best is None else min(best, s)
    nominal = 152 * 128 * 2 * 2070e6 / 1e12
    return {"tflops": round(flops / best / 1e12, 2), "seconds": round(best, 6), "flops": flops,
            "nominal_tflops": round(nominal, 1),
            "how": "lin_probe_ffma: SMs x 4 CTAs x 256 threads, 8 independent fmaf chains each, best of 5 "
                   "(CUDA events)"}


# --------------------------------------------------------------- our arm

class LayerBench:
    """One layer on the device: inputs, rotating W copies, output, the full
    oracle result, and the three ways of calling it."""

    def __init__(self, torch, tll, oracle, layer, ctx, dev, stream, flush_buf, world=1, want_chain=False):
        self.torch, self.tll, self.layer, self.ctx, self.dev, self.stream = torch, tll, layer, ctx, dev, stream
        self.prec = PREC_NAME[layer.precision]
        self.dt = torch.bfloat16 if layer.in_bf16 else torch.float32
        self.esz = 2 if layer.in_bf16 else 4
        self.epi = "gelu" if layer.epilogue else "none"
        props = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(props, "L2_cache_size", 126 << 20))
        X, W, b = si.make_inputs(layer)
        self.X, self.W, self.b = X, W, b
        self.x = torch.from_numpy(X).to(dev).to(self.dt)
        w0 = torch.from_numpy(W).to(dev).to(self.dt)
        self.bias = None if b is None else torch.from_numpy(b).to(dev)
        self.w_bytes = layer.N * layer.K * self.esz
        n = max(2, math.ceil(4 * self.l2 / self.w_bytes))
        n += n % 2  # even: the chained mode alternates two activation buffers
        while n > 2 and n * self.w_bytes > (8 << 30):
            n -= 2
        self.n_copies = n
        self.ws = [w0] + [w0.clone() for _ in range(n - 1)]
        self.y = torch.empty((layer.M, layer.N), dtype=self.dt, device=dev)
        self.xp, self.yp = self.x.data_ptr(), self.y.data_ptr()
        self.bp = None if self.bias is None else self.bias.data_ptr()
        self.wps = [t.data_ptr() for t in self.ws]
        self.chain = None
        if want_chain and layer.N == layer.K:
            # Two activation buffers: call i reads buf[i % 2] and writes buf[(i + 1) % 2].
            self.chain = [self.x.clone(), torch.empty_like(self.x)]
        self.world = world
        self.timer = {}
        self.flush_buf = flush_buf
        self.oracle = oracle
        self.ref = None

    # one call of each kind (i = position in the sequence)
    def _call(self, xp, wp, yp):
        L = self.layer
        rc = self.ctx.forward_ptr(L.M, L.N, L.K, xp, wp, self.bp, yp, self.epi, self.prec, self.stream.cuda_stream)
        if rc != 0:
            raise self.tll.LinError(rc, "lin_forward")

    def step_independent(self, i):
        self._call(self.xp, self.wps[i % self.n_copies], self.yp)

    def step_chained(self, i):
        a, b = self.chain[i % 2], self.chain[(i + 1) % 2]
        self._call(a.data_ptr(), self.wps[i % self.n_copies], b.data_ptr())

    def parity(self):
        """Full-output parity of one call against the oracle (all M x N)."""
        torch, oracle = self.torch, self.oracle
        with torch.cuda.stream(self.stream):
            self.step_independent(0)
        self.stream.synchronize()
        self.ctx.check(self.stream)
        self.ref = oracle.linear(self.X, self.W, self.b, bool(self.layer.epilogue))
        got = self.y.float().cpu().numpy().astype(np.float64)
        err = oracle.rel_err(got, self.ref)
        tol = oracle.TOL[self.layer.precision]
        if not (np.all(np.isfinite(got)) and err <= tol):
            raise SystemExit(f"correctness gate failed for {self.layer.name}: rel_err {err} > {tol}")
        return err, tol

    def parity_after(self):
        got = self.y.float().cpu().numpy().astype(np.float64)
        return self.oracle.rel_err(got, self.ref)

    def chain_parity(self):
        """Two chained calls: each output against the oracle applied to the
        exact values the call read (the previous call's bf16 output)."""
        torch, oracle = self.torch, self.oracle
        a0 = self.chain[0].float().cpu().numpy()
        with torch.cuda.stream(self.stream):
            self.step_chained(0)
            self.step_chained(1)
        self.stream.synchronize()
        self.ctx.check(self.stream)
        y1 = self.chain[1].float().cpu().numpy()
        y2 = self.chain[0].float().cpu().numpy()
        e1 = oracle.rel_err(y1.astype(np.float64), oracle.linear(a0, self.W, self.b, bool(self.layer.epilogue)))
        e2 = oracle.rel_err(y2.astype(np.float64), oracle.linear(y1, self.W, self.b, bool(self.layer.epilogue)))
        tol = oracle.TOL[self.layer.precision]
        if not (e1 <= tol and e2 <= tol):
            raise SystemExit(f"chained calls are wrong for {self.layer.name}: rel_err {e1}, {e2} > {tol}")
        # Restore buffer 0 to X for the timed chain (its values do not change the work).
        self.chain[0].copy_(self.x)
        torch.cuda.synchronize()
        return max(e1, e2)

    def mode(self, name, early_level, step):
        torch = self.torch
        self.ctx.set_option(self.tll.OPT_EARLY_START, early_level)
        # Warm-up in this mode (attributes set, the stream's last output known).
        with torch.cuda.stream(self.stream):
            for i in range(3):
                step(i)
        self.stream.synchronize()
        if name not in self.timer:
            self.timer[name] = CallTimer(torch, self.stream, step, self.n_copies, self.flush_buf, self.world)
        return self.timer[name]

    def time_mode(self, name, early_level, step, steps, steady=True):
        """{"seconds": exactly `steps` calls, "steady_s_per_call": over a
        longer run, "fill_drain_us", "plan"} for one way of calling."""
        t = self.mode(name, early_level, step)
        secs = t.measure(steps)
        plan = self.ctx.last_plan()
        out = {"seconds": secs, "calls": steps, "plan": plan}
        if steady:
            n_long = steady_calls(secs / steps, steps)
            if n_long > steps:
                long_s = t.measure(n_long)
                out["steady_s_per_call"] = long_s / n_long
                out["steady_calls"] = n_long
            else:
                out["steady_s_per_call"] = secs / steps
                out["steady_calls"] = steps
            out["fill_drain_us"] = round((secs - steps * out["steady_s_per_call"]) * 1e6, 3)
        return out

    def value_of(self, s_per_call):
        L = self.layer
        if is_hbm_bound(L):
            return L.algorithmic_bytes() / s_per_call / 1e9, "GB/s"
        return L.flops / s_per_call / 1e12, "TFLOP/s"


def plan_dict(plan):
    return {k: v for k, v in plan.as_dict().items() if k != "kernel_name"}


def mode_summary(lb: LayerBench, m, peaks, src, ffma, traffic=None):
    per_call = m["seconds"] / m["calls"]
    v, unit = lb.value_of(per_call)
    roof = roofline_for(lb.layer, per_call, peaks, src, traffic, ffma)
    d = {"value": round(v, 3), "unit": unit, "ms_per_step": round(per_call * 1e3, 6), "frac": roof["frac"],
         "kernel": m["plan"].as_dict()["kernel_name"], "plan": plan_dict(m["plan"])}
    if "steady_s_per_call" in m:
        sv, _ = lb.value_of(m["steady_s_per_call"])
        d["steady"] = {"value": round(sv, 3), "ms_per_step": round(m["steady_s_per_call"] * 1e3, 6),
                       "calls": m["steady_calls"]}
        d["fill_drain_us"] = m["fill_drain_us"]
    return d


def per_config_entries(torch, tll, oracle, ctx, dev, stream, flush_buf, peaks, src, ffma, done=None):
    """Every benchmark configuration, isolated and back to back, with its
    full-output parity against the oracle."""
    out = []
    for layer in PER_CONFIG:
        if done and layer.name in done:
            out.append(done[layer.name])
            continue
        t0 = time.perf_counter()
        lb = LayerBench(torch, tll, oracle, layer, ctx, dev, stream, flush_buf)
        err, tol = lb.parity()
        rate = 50e12 if layer.precision == si.PREC_FP32 else 1e15
        guess = max(layer.flops / rate, layer.algorithmic_bytes() / 6e12, 3e-6)
        n = max(20, min(2000, int(0.02 / guess)))
        iso = lb.time_mode("isolated", tll.EARLY_NONE, lb.step_independent, n, steady=False)
        b2b = lb.time_mode("back_to_back", tll.EARLY_ALL, lb.step_independent, n, steady=False)
        err_after = lb.parity_after()
        if not err_after <= tol:
            raise SystemExit(f"{layer.name}: output after the timed calls is wrong (rel_err {err_after})")
        e = {"workload": layer.name, "M": layer.M, "N": layer.N, "K": layer.K, "precision": lb.prec,
             "epilogue": lb.epi, "bias": layer.bias, "bound": "hbm" if is_hbm_bound(layer) else
             ("alu" if layer.precision == si.PREC_FP32 else "tensor"),
             "isolated": mode_summary(lb, iso, peaks, src, ffma),
             "back_to_back": mode_summary(lb, b2b, peaks, src, ffma),
             "rel_err": err, "rel_err_after_timed_calls": err_after, "tol": tol,
             "compared": f"all {layer.M * layer.N} outputs", "calls_timed": n,
             "w_copies": lb.n_copies}
        out.append(e)
        log(f"per_config {layer.name}: isolated {e['isolated']['value']} {e['isolated']['unit']} "
            f"({e['isolated']['frac']}), back to back {e['back_to_back']['value']} ({e['back_to_back']['frac']}), "
            f"rel_err {err:.2e} [{time.perf_counter() - t0:.1f} s]")
        del lb
        torch.cuda.empty_cache()
    return out


def bench_ours(layer: si.Layer, steps: int, warmup: int, world: int, rank: int, local_rank: int,
               with_cpu_baseline: bool, e2e_steps: int, with_per_config: bool):
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ctx = tll.Context(local_rank)
    stream = torch.cuda.Stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    flush_buf = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    peaks, src = load_peaks()
    ffma = measure_ffma_peak(torch, ctx, dev, stream)
    log(f"ffma probe: {ffma['tflops']} TFLOP/s (nominal {ffma['nominal_tflops']})")

    lb = LayerBench(torch, tll, oracle, layer, ctx, dev, stream, flush_buf, world, want_chain=True)
    err, tol = lb.parity()
    chain_err = lb.chain_parity() if lb.chain is not None else None
    for i in range(max(warmup, 3)):
        lb.step_independent(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    b2b_t = lb.mode("back_to_back", tll.EARLY_ALL, lb.step_independent)
    b2b_t.measure(steps)  # prepares and warms the graphs
    b2b_t.soak(1.0)
    b2b = lb.time_mode("back_to_back", tll.EARLY_ALL, lb.step_independent, steps)
    clocks = sampler.stop()
    ctx.check(stream)
    err_after = lb.parity_after()
    if not err_after <= tol:
        raise SystemExit(f"output after the timed steps is wrong for {layer.name}: rel_err {err_after} > {tol}")
    iso = lb.time_mode("isolated", tll.EARLY_NONE, lb.step_independent, steps)
    chained = None
    if lb.chain is not None:
        chained = lb.time_mode("chained", tll.EARLY_WEIGHTS, lb.step_chained, steps)
    ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)

    unit_bytes = layer.algorithmic_bytes()
    local_s = b2b["seconds"]
    max_s, total_units = aggregate(local_s, float(steps) * unit_bytes, world, dev)
    per_launch_s = local_s / steps
    if is_hbm_bound(layer):
        value, unit = total_units / max_s / 1e9, "GB/s"
    else:
        value, unit = world * steps * layer.flops / max_s / 1e12, "TFLOP/s"
    plan = b2b["plan"]
    kfile = {tll.KERNEL_SKINNY: "skinny.cu", tll.KERNEL_FFMA: "ffma.cu", tll.KERNEL_TC: "tc.cu",
             tll.KERNEL_GEMV: "gemv.cu"}.get(plan.kernel)
    traffic = traffic_from_profile(kfile, layer.name) if kfile else None
    roof = roofline_for(layer, per_launch_s, peaks, src, traffic, ffma)

    # End to end through the public API with host buffers: pinned host X, W,
    # bias in, Y out, every step, copies inside the timed region, the
    # library's default early start (the inputs arrive by host copies on the
    # same stream, which the library does not track).
    dt, esz = lb.dt, lb.esz
    hx = torch.from_numpy(lb.X).to(dt).pin_memory()
    hw = torch.from_numpy(lb.W).to(dt).pin_memory()
    hb = None if lb.b is None else torch.from_numpy(lb.b).pin_memory()
    hy = torch.empty((layer.M, layer.N), dtype=dt).pin_memory()
    dx, dw = torch.empty_like(lb.x), torch.empty_like(lb.ws[0])
    db = None if lb.bias is None else torch.empty_like(lb.bias)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        if db is not None:
            db.copy_(hb, non_blocking=True)
        out = tll.forward(dx, dw, db, epilogue=lb.epi, precision=lb.prec, ctx=ctx)
        hy.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        stream.synchronize()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_err = oracle.rel_err(hy.float().numpy().astype(np.float64), lb.ref)
    if not e2e_err <= tol:
        raise SystemExit(f"end-to-end output is wrong for {layer.name}: rel_err {e2e_err}")
    h2d = hx.numel() * esz + hw.numel() * esz + (0 if hb is None else hb.numel() * 4)
    d2h = hy.numel() * esz
    e2e_val = unit_bytes / e2e_s / 1e9 if unit == "GB/s" else layer.flops / e2e_s / 1e12
    e2e = {"value": round(e2e_val * world, 3), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": e2e_steps, "api": "transformer_linear_layer_gb300.forward (C ABI lin_forward)",
           "rel_err": e2e_err}

    cpu = None
    if with_cpu_baseline and rank == 0:
        cpu = cpu_baseline(layer, lb.X, lb.W, lb.b, unit)

    per_cfg = None
    if with_per_config and rank == 0:
        del hx, hw, hy, dx, dw
        per_cfg = per_config_entries(torch, tll, oracle, ctx, dev, stream, flush_buf, peaks, src, ffma)

    b2b_sum = mode_summary(lb, b2b, peaks, src, ffma, traffic)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(max_s / steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": lb.prec, "data": "synthetic",
        "config": {"workload": layer.name, "M": layer.M, "N": layer.N, "K": layer.K,
                   "bias": layer.bias, "epilogue": lb.epi, "precision": lb.prec,
                   "kernel": plan.as_dict()["kernel_name"], "plan": plan_dict(plan),
                   "l2": f"cold W: {lb.n_copies} rotating copies of W ({lb.n_copies * lb.w_bytes >> 20} MiB > L2 "
                         f"{l2 >> 20} MiB) and a read of {2 * l2 >> 20} MiB before each timed region; exactly "
                         f"`steps` calls replayed from warm CUDA graphs",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "parity_gate": {"rel_err": err, "rel_err_after_timed_steps": err_after, "tol": tol,
                                   "compared": f"all {layer.M * layer.N} outputs",
                                   "chained_rel_err": chain_err},
                   "steps_are": "independent back-to-back calls (same X, rotating W copies) with the early start "
                                "at level 2 (LIN_OPT_EARLY_START): a call may start and read its inputs before its "
                                "predecessor finishes and writes Y after it; isolated_call and e2e use the library "
                                "default (off), chained_call level 1 with X = the previous call's Y"},
        "back_to_back": b2b_sum,
        "isolated_call": dict(mode_summary(lb, iso, peaks, src, ffma),
                              note="early start off (the library default): each call waits for the previous kernel "
                                   "to finish before it reads anything"),
        "chained_call": None if chained is None else dict(
            mode_summary(lb, chained, peaks, src, ffma),
            note="X of call i+1 = Y of call i; early start level 1: W streams before the wait, X after it"),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "ffma_peak": ffma,
        "gpu_launches": steps * (0 if plan.kernel in (tll.KERNEL_NONE,) else 1),
        "per_config": per_cfg,
    }
    ctx.close()
    return line


# ---------------------------------------------------------------- backward

class BwdWork:
    """A backward GEMM of a layer or a fused forward: which 1 is dX = dZ W
    (M x K, reduction N), 2 is dW = dZ^T X (N x K, reduction M), 3 is dX
    carried through the previous layer's GELU, (dZ W) * gelu'(Zp) (reads Zp,
    M x K, too), 4 is the forward with the residual add in its store,
    Y = X W^T + bias + R (reads R, M x N)."""

    COMPUTES = {1: "dX = dZ W", 2: "dW = dZ^T X", 3: "dZp = (dZ W) * gelu'(Zp)", 4: "Y = X W^T + bias + R"}

    def __init__(self, name, which, M, N, K, precision):
        self.name, self.which, self.M, self.N, self.K, self.precision = name, which, M, N, K, precision
        self.flops = 2.0 * M * N * K

    def algorithmic_bytes(self):
        esz = 2 if self.precision == si.PREC_BF16 else 4
        M, N, K = self.M, self.N, self.K
        if self.which == 4:  # X, W, R and Y once each, plus the fp32 bias
            return (M * K + N * K + 2 * M * N) * esz + 4 * N
        other = N * K if self.which in (1, 3) else M * K   # W or X
        out = M * K if self.which in (1, 3) else N * K     # dX or dW
        extra = M * K if self.which == 3 else 0            # Zp
        return (M * N + other + out + extra) * esz


BWD_WORKLOADS = [BwdWork(f"{base}_{'dx' if which == 1 else 'dw'}", which, M, N, K, prec)
                 for base, M, N, K, prec in (("gpt2_fc1_m8192_bf16", 8192, 3072, 768, si.PREC_BF16),
                                             ("gpt2_fc2_m8192_bf16", 8192, 768, 3072, si.PREC_BF16),
                                             ("gpt2_fc1_m128_fp32", 128, 3072, 768, si.PREC_FP32),
                                             ("gpt2_fc2_m128_fp32", 128, 768, 3072, si.PREC_FP32))
                 for which in (1, 2)] + [
    BwdWork("gpt2_fc2_m8192_bf16_dx_gelu", 3, 8192, 768, 3072, si.PREC_BF16),
    BwdWork("gpt2_fc2_m128_fp32_dx_gelu", 3, 128, 768, 3072, si.PREC_FP32),
    BwdWork("gpt2_proj_m8192_bf16_residual", 4, 8192, 768, 768, si.PREC_BF16),
    BwdWork("gpt2_fc2_m8192_bf16_residual", 4, 8192, 768, 3072, si.PREC_BF16),
    BwdWork("gpt2_proj_m128_fp32_residual", 4, 128, 768, 768, si.PREC_FP32)]


def bench_backward(work: BwdWork, steps: int, warmup: int, world: int, rank: int, local_rank: int):
    """Back-to-back backward GEMMs or fused forwards through the C ABI
    (lin_backward_data, lin_backward_weight, lin_backward_data_gelu,
    lin_forward_residual), the streamed operand (dZ, or W for the forward)
    rotating over copies larger than L2, exactly `steps` calls replayed from
    warm CUDA graphs; full-output parity gate against the oracle."""
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ctx = tll.Context(local_rank)
    ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_ALL)  # library calls back to back only
    lib = tll.library()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    prec = PREC_NAME[work.precision]
    dt = torch.bfloat16 if work.precision == si.PREC_BF16 else torch.float32
    esz = 2 if work.precision == si.PREC_BF16 else 4
    M, N, K = work.M, work.N, work.K
    rnd = si.round_bf16 if work.precision == si.PREC_BF16 else (lambda a: a)
    if work.which == 4:  # forward: "dZ" is X (M x K), B is W (N x K), plus bias and the residual R
        dZ = rnd(si.normal(31, 1, (M, K)))
        B = rnd(si.normal(31, 2, (N, K), 0.0, 0.02))
        R = rnd(si.normal(31, 4, (M, N)))
        bias_h = si.normal(31, 5, (N,), 0.0, 0.02)
        bias_d = torch.from_numpy(bias_h).to(dev)
        r_dev = torch.from_numpy(R).to(dev).to(dt)
    else:
        dZ = rnd(si.normal(31, 1, (M, N), 0.0, 0.1))
        B = rnd(si.normal(31, 2, (N, K), 0.0, 0.02) if work.which in (1, 3) else si.normal(31, 3, (M, K)))
        if work.which == 3:
            Zp = rnd(si.normal(31, 4, (M, K)))
            zp_dev = torch.from_numpy(Zp).to(dev).to(dt)
    dz0 = torch.from_numpy(dZ).to(dev).to(dt)
    b_dev = torch.from_numpy(B).to(dev).to(dt)
    rot0 = b_dev if work.which == 4 else dz0  # the operand streamed from HBM every step
    rot_bytes = rot0.numel() * esz
    n_copies = max(2, math.ceil(4 * l2 / rot_bytes))
    while n_copies > 2 and n_copies * rot_bytes > (8 << 30):
        n_copies -= 1
    rots = [rot0] + [rot0.clone() for _ in range(n_copies - 1)]
    out = torch.empty((M, N) if work.which == 4 else ((M, K) if work.which in (1, 3) else (N, K)), dtype=dt,
                      device=dev)
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream

    def step(i):
        r = rots[i % n_copies].data_ptr()
        if work.which == 1:
            rc = lib.lin_backward_data(ctx._h, M, N, K, r, b_dev.data_ptr(), out.data_ptr(), work.precision, sptr)
        elif work.which == 2:
            rc = lib.lin_backward_weight(ctx._h, M, N, K, r, b_dev.data_ptr(), out.data_ptr(), None,
                                         work.precision, sptr)
        elif work.which == 3:
            rc = lib.lin_backward_data_gelu(ctx._h, M, N, K, r, b_dev.data_ptr(), zp_dev.data_ptr(), out.data_ptr(),
                                            work.precision, sptr)
        else:
            rc = lib.lin_forward_residual(ctx._h, M, N, K, dz0.data_ptr(), r, bias_d.data_ptr(), r_dev.data_ptr(),
                                          out.data_ptr(), 0, work.precision, sptr)
        if rc != 0:
            raise tll.LinError(rc, work.COMPUTES[work.which])

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    ctx.check(stream)
    if work.which == 1:
        ref = oracle.backward_dx(dZ, B)
    elif work.which == 2:
        ref, _ = oracle.backward_dw(dZ, B, with_bias=False)
    elif work.which == 3:
        ref = oracle.backward_dx_gelu(dZ, B, Zp)
    else:
        ref = oracle.linear_residual(dZ, B, R, bias_h)
    err = oracle.rel_err(out.float().cpu().numpy().astype(np.float64), ref)
    tol = oracle.TOL[si.PREC_BF16] if work.precision == si.PREC_BF16 else oracle.TOL[si.PREC_FP32]
    if not err <= tol:
        raise SystemExit(f"correctness gate failed for {work.name}: rel_err {err} > {tol}")

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    stream.synchronize()
    flush_buf = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    timer = CallTimer(torch, stream, step, n_copies, flush_buf, world)
    timer.measure(steps)
    sampler = ClockSampler(local_rank)
    timer.soak(1.0)
    local_s = timer.measure(steps)
    clocks = sampler.stop()
    ctx.check(stream)
    err_after = oracle.rel_err(out.float().cpu().numpy().astype(np.float64), ref)
    if not err_after <= tol:
        raise SystemExit(f"output after the timed steps is wrong for {work.name}: rel_err {err_after} > {tol}")
    max_s, _ = aggregate(local_s, float(steps) * work.algorithmic_bytes(), world, dev)
    peaks, src = load_peaks()
    roof = roofline_for(work, local_s / steps, peaks, src, None)
    line = {
        "metric": METRIC, "value": round(world * steps * work.flops / max_s / 1e12, 3), "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": round(max_s / steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": prec, "data": "synthetic",
        "config": {"workload": work.name, "M": M, "N": N, "K": K,
                   "computes": work.COMPUTES[work.which],
                   "kernel": tll.KERNEL_NAMES[ctx.last_plan().kernel] if work.which == 4 else
                   ("tc (MN-major operands)" if work.precision == si.PREC_BF16 else "bwd_ffma"),
                   "l2": f"cold {'W' if work.which == 4 else 'dZ'}: {n_copies} rotating copies "
                         f"({n_copies * rot_bytes >> 20} MiB > L2 {l2 >> 20} MiB), exactly `steps` calls "
                         f"replayed from warm CUDA graphs",
                   "parity_gate": {"rel_err": err, "rel_err_after_timed_steps": err_after, "tol": tol,
                                   "compared": f"all {out.numel()} outputs"}},
        "roofline": roof, "clocks": clocks, "gpu_launches": steps,
    }
    ctx.close()
    return line


# ---------------------------------------------------------------- attention

ATTN_WORKLOADS = {si.GPT2_ATTN_B64.name: si.GPT2_ATTN_B64}


def attention_bound(att, qkv, out, scale):
    """Per-element bound on |out - oracle| from the kernel's arithmetic: P
    rounded to bf16 (relative error at most 2^-8) before its product with v,
    the output rounded to bf16 (2^-8), fp32 sums:
    1.05 * 2^-8 (sum_j p_ij |v_j| + |out_ref|) + 1e-5."""
    B, T, H, D = att.B, att.T, att.H, att.D
    x = qkv.astype(np.float64).reshape(B, T, 3, H, D)
    s = np.einsum("bihd,bjhd->bhij", x[:, :, 0], x[:, :, 1]) * scale
    if att.causal:
        s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    a = np.einsum("bhij,bjhd->bihd", p, np.abs(x[:, :, 2])).reshape(B * T, H * D)
    return 1.05 * 2.0 ** -8 * (a + np.abs(out)) + 1e-5


def bench_attention(att, steps: int, warmup: int, world: int, rank: int, local_rank: int, cpu: bool = True):
    """Back-to-back fused attention forwards through the C ABI
    (lin_attention_forward), the qkv input rotating over copies larger than
    L2, exactly `steps` calls replayed from warm CUDA graphs; every output
    element checked against the oracle before and after the timed calls."""
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ctx = tll.Context(local_rank)
    lib = tll.library()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    qkv = si.make_qkv(att)
    scale = 1.0 / math.sqrt(att.D)
    q0 = torch.from_numpy(qkv).to(dev).to(torch.bfloat16)
    in_bytes = q0.numel() * 2
    n_copies = max(2, math.ceil(4 * l2 / in_bytes))
    rots = [q0] + [q0.clone() for _ in range(n_copies - 1)]
    out = torch.empty((att.B * att.T, att.C), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream

    def step(i):
        rc = lib.lin_attention_forward(ctx._h, att.B, att.T, att.H, att.D, rots[i % n_copies].data_ptr(),
                                       out.data_ptr(), None, int(att.causal), 0.0, sptr)
        if rc != 0:
            raise tll.LinError(rc, "lin_attention_forward")

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    ctx.check(stream)
    ref = oracle.attention(qkv, att.B, att.T, att.H, att.D, causal=att.causal, scale=scale)
    bound = attention_bound(att, qkv, ref, scale)

    def gate(what):
        got = out.float().cpu().numpy().astype(np.float64)
        r = float(np.max(np.abs(got - ref) / bound))
        if not r <= 1.0:
            raise SystemExit(f"{what} for {att.name}: max |out - oracle| / bound = {r}")
        return r

    err = gate("correctness gate failed")
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    stream.synchronize()
    flush_buf = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    timer = CallTimer(torch, stream, step, n_copies, flush_buf, world)
    timer.measure(steps)
    sampler = ClockSampler(local_rank)
    timer.soak(1.0)
    local_s = timer.measure(steps)
    clocks = sampler.stop()
    ctx.check(stream)
    err_after = gate("output after the timed steps is wrong")
    byts = att.algorithmic_bytes()
    max_s, total = aggregate(local_s, float(steps) * byts, world, dev)
    peaks, src = load_peaks()
    per = local_s / steps
    ach = byts / per / 1e9
    tflops = att.flops / per / 1e12
    roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4),
            "traffic": traffic_from_profile("attn.cu", att.name, kernel="attn_fwd_kernel"),
            "peak_source": f"hbm copy, {src}",
            "algorithmic_bytes_per_launch": byts,
            "tensor": {"achieved_tflops": round(tflops, 2), "peak": peaks["bf16_tflops"],
                       "frac": round(tflops / peaks["bf16_tflops"], 4),
                       "algorithmic_flops_per_launch": att.flops}}
    cpu_line = None
    if cpu and rank == 0 and world == 1:
        cores = oracle.max_threads()
        nb = max(1, min(att.B, 4))
        sub = qkv[:nb * att.T]
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.attention(sub, nb, att.T, att.H, att.D, causal=att.causal, scale=scale, nthreads=cores)
            reps += 1
            el = time.perf_counter() - t0
            if el >= 10.0 or reps >= 1000:
                break
        per_cpu = el / reps * att.B / nb
        cpu_line = {"value": round(byts / per_cpu / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                    "sample": f"{reps} x oracle attention on {nb} of {att.B} sequences ({el:.1f} s), scaled to "
                              f"the whole batch"}
    line = {
        "metric": METRIC, "value": round(total / max_s / 1e9, 3), "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": round(max_s / steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": att.name, "B": att.B, "T": att.T, "H": att.H, "D": att.D, "causal": att.causal,
                   "computes": "out = softmax(q k^T / sqrt(D)) v per head, q/k/v read from the qkv projection's "
                               "(B*T) x 3C output", "kernel": "attn_fwd_kernel",
                   "tflops": round(world * steps * att.flops / max_s / 1e12, 3),
                   "l2": f"cold qkv: {n_copies} rotating copies ({n_copies * in_bytes >> 20} MiB > L2 "
                         f"{l2 >> 20} MiB), exactly `steps` calls replayed from warm CUDA graphs",
                   "parity_gate": {"max_err_over_bound": err, "after_timed_steps": err_after,
                                   "bound": "1.05 * 2^-8 (sum_j p_ij |v_j| + |ref|) + 1e-5 per element",
                                   "compared": f"all {out.numel()} outputs"}},
        "roofline": roof, "cpu_baseline": cpu_line, "clocks": clocks, "gpu_launches": steps,
    }
    ctx.close()
    return line


def cpu_baseline(layer: si.Layer, X, W, b, unit, budget_s=10.0):
    """The oracle as it stands on the host cores: whole layers when one takes
    under a second, else a seeded sample of rows, repeated for ~budget_s."""
    import oracle

    cores = oracle.max_threads()
    per_row_macs = layer.N * layer.K
    rows = layer.M
    # estimate ~0.5 G MAC/s per core; keep one call under ~2 s
    if per_row_macs * rows > 1e9 * cores:
        rows = max(1, int(1e9 * cores // per_row_macs))
    Xs = X[:rows]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.linear(Xs, W, b, bool(layer.epilogue), nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    per_call = el / reps
    frac = rows / layer.M
    per_layer = per_call / frac
    if unit == "GB/s":
        v = layer.algorithmic_bytes() / per_layer / 1e9
    else:
        v = layer.flops / per_layer / 1e12
    sample = (f"{reps} x oracle on {'all' if rows == layer.M else rows} of {layer.M} rows "
              f"({el:.1f} s), scaled to one whole layer")
    return {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}


# --------------------------------------------------------- reference arm

def bench_reference(layer: si.Layer, steps: int, warmup: int):
    import oracle

    X, W, b = si.make_inputs(layer)
    unit = "GB/s" if is_hbm_bound(layer) else "TFLOP/s"
    cores = oracle.max_threads()
    # Each step: the oracle on a bounded sample of rows (whole layer when small).
    rows = layer.M
    per_row_macs = layer.N * layer.K
    if per_row_macs * rows > 2e8 * cores:
        rows = max(1, int(2e8 * cores // per_row_macs))
    Xs = X[:rows]
    for _ in range(warmup):
        oracle.linear(Xs, W, b, bool(layer.epilogue), nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.linear(Xs, W, b, bool(layer.epilogue), nthreads=cores)
    el = (time.perf_counter() - t0) / steps
    per_layer = el * layer.M / rows
    v = layer.algorithmic_bytes() / per_layer / 1e9 if unit == "GB/s" else layer.flops / per_layer / 1e12
    sample = f"oracle on {'all' if rows == layer.M else rows} of {layer.M} rows per step, scaled to one layer"
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit, "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": round(el * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": layer.name, "M": layer.M, "N": layer.N, "K": layer.K, "bias": layer.bias,
                   "epilogue": "gelu" if layer.epilogue else "none", "precision": PREC_NAME[layer.precision]},
        "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def bench_reference_attention(att, steps: int, warmup: int):
    """The oracle's attention timed on the host cores: each step computes a
    bounded sample of the batch (whole sequences), scaled to the whole batch."""
    import oracle

    cores = oracle.max_threads()
    qkv = si.make_qkv(att)
    nb = max(1, min(att.B, 2))
    sub = qkv[:nb * att.T]
    scale = 1.0 / math.sqrt(att.D)
    for _ in range(warmup):
        oracle.attention(sub, nb, att.T, att.H, att.D, causal=att.causal, scale=scale, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.attention(sub, nb, att.T, att.H, att.D, causal=att.causal, scale=scale, nthreads=cores)
    el = (time.perf_counter() - t0) / steps
    per_batch = el * att.B / nb
    v = att.algorithmic_bytes() / per_batch / 1e9
    sample = f"oracle attention on {nb} of {att.B} sequences per step, scaled to the whole batch"
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": round(el * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": att.name, "B": att.B, "T": att.T, "H": att.H, "D": att.D, "causal": att.causal},
        "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------- ncu

def profile_launches(name: str, n: int) -> int:
    """A small, self-contained launch sequence for a profiler: the workload's
    inputs, one call checked against the oracle, then n independent calls on
    rotating W copies (the library's default launch mode), synchronised. The
    launches to capture are the last n."""
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    dev = torch.device("cuda", 0)
    ctx = tll.Context(0)
    stream = torch.cuda.Stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    flush = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    if name in BWD_BY_NAME:
        raise SystemExit("--profile-launches covers forward workloads and attention")
    if name in ATTN_WORKLOADS:
        att = ATTN_WORKLOADS[name]
        dq = torch.from_numpy(si.make_qkv(att)).to(dev).to(torch.bfloat16)
        qs = [dq] + [dq.clone() for _ in range(3)]
        out = torch.empty((att.B * att.T, att.C), dtype=torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            for i in range(n + 1):
                torch.sum(flush, dim=0)
                tll.attention_forward(qs[i % 4], att.B, att.T, att.H, causal=att.causal, out=out, ctx=ctx,
                                      stream=stream)
        stream.synchronize()
        ctx.check(stream)
        log(f"{name}: {n + 1} launches of attn_fwd_kernel")
        ctx.close()
        return 0
    lb = LayerBench(torch, tll, oracle, WORKLOADS[name], ctx, dev, stream, flush)
    err, tol = lb.parity()
    with torch.cuda.stream(stream):
        for i in range(n):
            lb.step_independent(i + 1)
    stream.synchronize()
    ctx.check(stream)
    log(f"{name}: {n} launches of {ctx.last_plan().as_dict()['kernel_name']}, parity rel_err {err:.3e} (tol {tol})")
    ctx.close()
    return 0


# ---------------------------------------------------------------- timelines

TIMELINE_TC = ("gpt2_qkv_m8192_bf16", "gpt2_proj_m8192_bf16", "gpt2_fc1_m8192_bf16", "gpt2_fc2_m8192_bf16",
               "gpt2_lmhead_m8192_bf16")


def _med(a):
    return round(float(np.median(a)) / 1e3, 3) if len(a) else None


def timeline_report(which: str = "all") -> int:
    """Kernel timelines from the timeline build (stamps compiled in, see
    lin_timeline): one JSON line per case on stdout.

    tc: one cold launch (after an L2 flush) of each M = 8192 GPT-2 layer and
    the LM head, with the table's plan and with the SM-pair plan; per work
    item j (medians over CTAs, us): the MMA issue span (first MMA to the
    accumulator's commit), the epilogue span (accumulator ready to the last
    store issued, warps 2 and 9), the item's end, and the pace of K stages.
    skinny: four consecutive calls of the M = 16 layer in each calling mode;
    per call (us from the first CTA's start): first and last CTA start, median
    dependency-wait release, median first and last stage landed, last CTA
    done.
    attn: the fused attention forward on GPT-2's batched shape, one cold call
    and the last of 20 back-to-back calls; per CTA work item n (medians over
    CTAs, us from the first CTA's start) the stamps of lin_timeline's
    attention record, and per item the softmax group's chain: S seen to P
    released, P released to P.V issued (all four warps), P.V seen to output
    stored.
    `which` selects tc, skinny, attn or all."""
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    tll.use_timeline_build()
    dev = torch.device("cuda", 0)
    ctx = tll.Context(0)
    stream = torch.cuda.Stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    flush = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    sm = ctx.sm_count

    for name in (TIMELINE_TC if which in ("all", "tc") else ()):
        layer = WORKLOADS[name]
        lb = LayerBench(torch, tll, oracle, layer, ctx, dev, stream, flush)
        if name == TIMELINE_TC[0]:
            lb.parity()  # the stamped kernel computes what the library's does
        nkb = (layer.K * lb.esz + 127) // 128
        for variant in (None, 3):
            plan = ctx.plan(layer.M, layer.N, layer.K, lb.prec, lb.epi) if variant is None else \
                tll.plan_make(sm, tll.KERNEL_TC, variant, 0, layer.M, layer.N, layer.K, lb.prec)
            with torch.cuda.stream(stream):
                for i in range(3):
                    rc = ctx.forward_plan_ptr(plan, layer.M, layer.N, layer.K, lb.xp, lb.wps[i % lb.n_copies], lb.bp,
                                              lb.yp, lb.epi, lb.prec, stream.cuda_stream)
                    if rc != 0:
                        raise tll.LinError(rc, "lin_forward_plan")
                torch.sum(flush, dim=0, out=sink)
            stream.synchronize()
            tll.timeline_clear(tll.KERNEL_TC)
            with torch.cuda.stream(stream):
                ctx.forward_plan_ptr(plan, layer.M, layer.N, layer.K, lb.xp, lb.wps[3 % lb.n_copies], lb.bp, lb.yp,
                                     lb.epi, lb.prec, stream.cuda_stream)
            stream.synchronize()
            ctx.check(stream)
            t = tll.timeline(tll.KERNEL_TC)[:plan.grid_x]
            t0 = t[:, 0][t[:, 0] > 0].min()
            items = []
            for j in range(32):
                ms, mc, et, ed, e9 = t[:, 8 + 4 * j], t[:, 9 + 4 * j], t[:, 10 + 4 * j], t[:, 11 + 4 * j], t[:, 136 + j]
                mm = (ms > 0) & (mc > 0)
                ee = (et > 0) & (ed > 0) & (e9 > 0)
                if not ee.any():
                    break
                items.append({"j": j, "ctas": int(ee.sum()),
                              "mma_issue_us": _med((mc - ms)[mm]), "epilogue_us": _med((np.maximum(ed, e9) - et)[ee]),
                              "done_us": _med((np.maximum(ed, e9) - t0)[ee])})
            done = [it["done_us"] for it in items]
            pace = [round(done[i + 1] - done[i], 3) for i in range(len(done) - 1)]
            rec = {"timeline": "tc_kernel", "workload": name, "plan": plan_dict(plan), "k_stages": nkb,
                   "span_us": round(float(t[:, 2].max() - t0) / 1e3, 3), "items": items[:8],
                   "item_pace_us": pace[:8],
                   "stage_pace_us": [round(p / nkb, 4) for p in pace[:8]]}
            print(json.dumps(rec), flush=True)
        del lb
        torch.cuda.empty_cache()

    if which in ("all", "attn"):
        timeline_attention(torch, tll, ctx, dev, stream, flush, sink)
    if which not in ("all", "skinny"):
        ctx.close()
        return 0
    layer = WORKLOADS[DEFAULT_WORKLOAD]
    lb = LayerBench(torch, tll, oracle, layer, ctx, dev, stream, flush, want_chain=True)
    lb.parity()
    for mode, level, step in (("isolated", tll.EARLY_NONE, lb.step_independent),
                              ("chained", tll.EARLY_WEIGHTS, lb.step_chained),
                              ("back_to_back", tll.EARLY_ALL, lb.step_independent)):
        ctx.set_option(tll.OPT_EARLY_START, level)
        with torch.cuda.stream(stream):
            for i in range(6):
                step(i)
        stream.synchronize()
        plan = ctx.last_plan()  # the plan this calling mode gets
        nblk = plan.grid_x * plan.grid_y
        ncall = max(1, min(4, tll.TIMELINE_CTAS // nblk))
        with torch.cuda.stream(stream):
            torch.sum(flush, dim=0, out=sink)
        stream.synchronize()
        tll.timeline_clear(tll.KERNEL_SKINNY)
        with torch.cuda.stream(stream):
            for i in range(ncall):
                step(6 + i)
        stream.synchronize()
        ctx.check(stream)
        t = tll.timeline(tll.KERNEL_SKINNY)[:nblk * ncall]
        t0 = t[:, 0][t[:, 0] > 0].min()
        calls = []
        for k in range(ncall):
            tk = t[k * nblk:(k + 1) * nblk]
            st = tk[:, 16:176]
            first = np.where(st > 0, st, np.iinfo(np.int64).max).min(axis=1)
            last = np.where(st > 0, st, 0).max(axis=1)
            r = lambda a: round(float(a - t0) / 1e3, 3)
            calls.append({"start_first": r(tk[:, 0].min()), "start_last": r(tk[:, 0].max()),
                          "wait_released": r(np.median(tk[:, 1])) if (tk[:, 1] > 0).all() else None,
                          "first_stage": r(np.median(first)),
                          "last_stage": r(np.median(last)), "last_stage_max": r(last.max()),
                          "done": r(tk[:, 3].max())})
        ends = [c["done"] for c in calls]
        print(json.dumps({"timeline": "skinny_kernel", "workload": layer.name, "mode": mode, "plan": plan_dict(plan),
                          "calls": calls, "call_to_call_us": [round(ends[i + 1] - ends[i], 3)
                                                              for i in range(len(ends) - 1)]}), flush=True)
    ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_NONE)
    ctx.close()
    return 0


def timeline_attention(torch, tll, ctx, dev, stream, flush, sink):
    att = si.GPT2_ATTN_B64
    q0 = torch.from_numpy(si.make_qkv(att)).to(dev).to(torch.bfloat16)
    qs = [q0] + [q0.clone() for _ in range(11)]
    out = torch.empty((att.B * att.T, att.C), dtype=torch.bfloat16, device=dev)
    sm = ctx.sm_count

    def call(i):
        tll.attention_forward(qs[i % len(qs)], att.B, att.T, att.H, causal=att.causal, out=out, ctx=ctx,
                              stream=stream)

    def report(mode):
        t = tll.timeline(tll.TIMELINE_ATTENTION)[:min(sm, att.B * att.H)]
        t0 = t[:, 0][t[:, 0] > 0].min()
        items = []
        for n in range(6):
            col = [t[:, 8 + 10 * n + k] for k in range(10)]
            if not (col[4] > 0).any():
                break
            med = [_med(c[c > 0] - t0) if (c > 0).any() else None for c in col]
            ok = (col[4] > 0) & (col[5] > 0) & (col[6] > 0) & (col[7] > 0) & (col[8] > 0)
            items.append({"n": n, "group": n % 2, "stamps_us": med,
                          "softmax_us": _med((col[5] - col[4])[ok]), "p_to_pv_us": _med((col[6] - col[5])[ok]),
                          "output_us": _med((col[8] - col[7])[ok])})
        print(json.dumps({"timeline": "attn_fwd_kernel", "workload": att.name, "mode": mode,
                          "setup_us": _med(t[:, 0] - t0), "wait_released_us": _med(t[:, 1] - t0),
                          "teardown_max_us": round(float(t[:, 2].max() - t0) / 1e3, 3), "items": items}), flush=True)

    with torch.cuda.stream(stream):
        call(0)
        torch.sum(flush, dim=0, out=sink)
    stream.synchronize()
    tll.timeline_clear(tll.TIMELINE_ATTENTION)
    with torch.cuda.stream(stream):
        call(1)
    stream.synchronize()
    ctx.check(stream)
    report("cold")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(20):
            call(i)
    g.replay()
    stream.synchronize()
    with torch.cuda.stream(stream):
        torch.sum(flush, dim=0, out=sink)
    stream.synchronize()
    tll.timeline_clear(tll.TIMELINE_ATTENTION)
    g.replay()
    stream.synchronize()
    ctx.check(stream)
    report("last of 20 back to back")


# ------------------------------------------------------------------- main

BWD_BY_NAME = {w.name: w for w in BWD_WORKLOADS}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(WORKLOADS) + sorted(BWD_BY_NAME) + sorted(ATTN_WORKLOADS))
    ap.add_argument("--all", action="store_true", help="one line per workload (stdout), default line last")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per_config section")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="for ncu: only a parity-checked call and this many plain launches of the workload "
                         "(no graphs, no timing), then exit")
    ap.add_argument("--timeline", nargs="?", const="all", default=None, choices=("all", "tc", "skinny", "attn"),
                    help="kernel timelines from the timeline build (JSON lines), then exit")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    steps, warmup = max(1, args.steps), max(3, args.warmup)

    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.workload in BWD_BY_NAME:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times forward workloads only"}))
            return 0
        if args.workload in ATTN_WORKLOADS:
            print(json.dumps(bench_reference_attention(ATTN_WORKLOADS[args.workload], min(steps, 200), warmup)),
                  flush=True)
            return 0
        ref_steps = min(steps, 200)
        line = bench_reference(WORKLOADS[args.workload], ref_steps, warmup)
        print(json.dumps(line), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    if args.profile_launches > 0:
        return profile_launches(args.workload, args.profile_launches)
    if args.timeline:
        return timeline_report(args.timeline)
    if args.workload in BWD_BY_NAME:
        work = BWD_BY_NAME[args.workload]
        line = bench_backward(work, steps, warmup, world, rank, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    if args.workload in ATTN_WORKLOADS:
        line = bench_attention(ATTN_WORKLOADS[args.workload], steps, warmup, world, rank, local_rank,
                               cpu=not args.no_cpu_baseline)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    names = [args.workload]
    if args.all:
        names = [n for n in WORKLOADS if n != args.workload] + [args.workload]
        for work in BWD_WORKLOADS:
            st = max(300, min(steps, int(2e13 / work.flops)))
            line = bench_backward(work, st, warmup, world, rank, local_rank)
            if rank == 0:
                print(json.dumps(line), flush=True)
        for att in ATTN_WORKLOADS.values():
            line = bench_attention(att, max(300, steps), warmup, world, rank, local_rank, cpu=False)
            if rank == 0:
                print(json.dumps(line), flush=True)
    for name in names:
        layer = WORKLOADS[name]
        default = name == args.workload
        # Other workloads: at least 300 steps and ~20 TFLOP.
        st = steps if default else max(300, min(steps, int(2e13 / max(layer.flops, 1e6))))
        line = bench_ours(layer, st, warmup, world, rank, local_rank,
                          with_cpu_baseline=(not args.no_cpu_baseline and default),
                          e2e_steps=args.e2e_steps if default else 5,
                          with_per_config=(default and not args.no_per_config and world == 1))
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
