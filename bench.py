"""Benchmark of the GB300 linear layer (one JSON line on stdout).

Default workload: the skinny linear layer, M = 16 vectors against a
4096 x 4096 bf16 weight stored out x in, fp32 accumulate, bf16 output, fp32
bias ("One multiply, one RTX 5090, eight kernels", "The multiply"). A step is
one call of the layer (dispatch, split-K stream of W, fixed-order reduction,
epilogue). Metric: achieved HBM GB/s over the algorithmic bytes (X + W + Y +
bias once each) with W cold: each step reads one of R identical copies of W
(R x 32 MiB > 4 x L2), so no step finds its W in L2 (the page's section
"Where the time goes" keeps its weights cold the same way, cycling through
copies of them).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --all]

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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


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


def roofline_for(layer: si.Layer, seconds_per_launch: float, peaks, peaks_src, traffic):
    """The bound that applies to this layer and the achieved fraction of it."""
    flops = layer.flops
    byts = layer.algorithmic_bytes()
    hbm = peaks["hbm_gbs"] * 1e9
    # Tensor peaks: bf16 measured; TF32 = bf16 x nominal ratio (1.1 / 2.25 PF dense).
    if layer.precision == si.PREC_BF16:
        tens, tens_note = peaks["bf16_tflops"] * 1e12, "bf16 dense, " + peaks_src
    elif layer.precision == si.PREC_TF32:
        tens, tens_note = peaks["bf16_tflops"] * 1e12 * (1.1 / 2.25), f"tf32 = bf16 {peaks_src} x 1.1/2.25 nominal"
    else:
        # FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock (nominal unit counts and clock)
        tens = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6
        tens_note = "fp32 FFMA = 152 SMs x 128 lanes x 2 x sm_max_mhz"
    t_mem, t_cmp = byts / hbm, flops / tens
    if t_mem >= t_cmp:
        ach = byts / seconds_per_launch / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"hbm copy, {peaks_src}", "algorithmic_bytes_per_launch": byts}
    ach = flops / seconds_per_launch / 1e12
    bound = "alu" if layer.precision == si.PREC_FP32 else "tensor"
    return {"bound": bound, "achieved": round(ach, 2), "peak": round(tens / 1e12, 1), "unit": "TFLOP/s",
            "frac": round(ach * 1e12 / tens, 4), "traffic": traffic, "peak_source": tens_note,
            "algorithmic_flops_per_launch": flops}


def traffic_from_profile(kernel_file: str, workload: str):
    """dram bytes per launch from the committed ncu summary of this kernel and
    workload (profiles/<kernel>_<workload>.md), or None when absent or when the
    kernel source has changed since the capture."""
    kernel = kernel_file.replace(".cu", "_kernel")
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


# --------------------------------------------------------------- our arm

def bench_ours(layer: si.Layer, steps: int, warmup: int, world: int, rank: int, local_rank: int,
               with_cpu_baseline: bool, e2e_steps: int):
    import torch

    import oracle
    import transformer_linear_layer_gb300 as tll

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ctx = tll.Context(local_rank)
    # The timed steps are library calls back to back and nothing else writes
    # their inputs on the stream: the programmatic early start is valid.
    ctx.set_option(tll.OPT_EARLY_START, tll.EARLY_ALL)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20))
    prec = PREC_NAME[layer.precision]
    dt = torch.bfloat16 if layer.in_bf16 else torch.float32
    esz = 2 if layer.in_bf16 else 4

    X, W, b = si.make_inputs(layer)
    x = torch.from_numpy(X).to(dev).to(dt)
    w0 = torch.from_numpy(W).to(dev).to(dt)
    bias = None if b is None else torch.from_numpy(b).to(dev)
    w_bytes = layer.N * layer.K * esz
    n_copies = max(2, math.ceil(4 * l2 / w_bytes))
    while n_copies > 2 and n_copies * w_bytes > (8 << 30):
        n_copies -= 1
    ws = [w0] + [w0.clone() for _ in range(n_copies - 1)]
    y = torch.empty((layer.M, layer.N), dtype=dt, device=dev)
    epi = "gelu" if layer.epilogue else "none"
    plan = ctx.plan(layer.M, layer.N, layer.K, prec, epi)

    # Correctness gate before any timing (full output for small layers, sampled otherwise).
    tll.forward(x, ws[-1], bias, epilogue=epi, precision=prec, out=y, ctx=ctx)
    torch.cuda.synchronize()
    ctx.check()
    if layer.M * layer.N * layer.K <= 1 << 31:
        ref = oracle.linear(X, W, b, bool(layer.epilogue))
        err = oracle.rel_err(y.float().cpu().numpy(), ref)
        gate = "full"
    else:
        rng = np.random.default_rng(1)
        ms, ns = rng.integers(0, layer.M, 512), rng.integers(0, layer.N, 512)
        ref = oracle.linear_entries(X, W, ms, ns, b, bool(layer.epilogue))
        got = y[torch.from_numpy(ms).to(dev), torch.from_numpy(ns).to(dev)].float().cpu().numpy()
        err = oracle.rel_err(got, ref)
        gate = "512 sampled outputs"
    tol = oracle.TOL[layer.precision]
    if not err <= tol:
        raise SystemExit(f"correctness gate failed for {layer.name}: rel_err {err} > {tol}")

    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    xp, yp = x.data_ptr(), y.data_ptr()
    bp = None if bias is None else bias.data_ptr()
    wps = [t.data_ptr() for t in ws]

    def step(i):
        # The public call (dispatch table, refined for back-to-back calls).
        rc = ctx.forward_ptr(layer.M, layer.N, layer.K, xp, wps[i % n_copies], bp, yp, epi, prec, sptr)
        if rc != 0:
            raise tll.LinError(rc, "lin_forward")

    # Warm-up (also sets kernel attributes before capture).
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    stream.synchronize()

    # CUDA graphs of G back-to-back steps (the launch tax is ~ the kernel time here).
    G = n_copies * max(1, 64 // n_copies)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                step(i)
        return g

    graph = capture(G)
    rem = steps % G
    graph_rem = capture(rem) if rem else None
    stream.synchronize()

    sampler = ClockSampler(local_rank)
    # Soak so the clock samples see the loaded state, then the timed region.
    soak_until = time.perf_counter() + 1.0
    with torch.cuda.stream(stream):
        while time.perf_counter() < soak_until:
            graph.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // G):
            graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    local_s = e0.elapsed_time(e1) / 1e3
    ctx.check(stream)
    plan = ctx.last_plan()  # the plan the timed calls ran with
    # The back-to-back steps overlap on the GPU; their result must still be right.
    if gate == "full":
        err_after = oracle.rel_err(y.float().cpu().numpy(), ref)
    else:
        got = y[torch.from_numpy(ms).to(dev), torch.from_numpy(ns).to(dev)].float().cpu().numpy()
        err_after = oracle.rel_err(got, ref)
    if not err_after <= tol:
        raise SystemExit(f"output after the timed steps is wrong for {layer.name}: rel_err {err_after} > {tol}")

    # The same call isolated: every call waits for the previous one to finish.
    ctx.set_option(tll.OPT_EARLY_START, 0)
    iso_steps = min(steps, 2000)
    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    g_iso = capture(min(G, iso_steps))
    with torch.cuda.stream(stream):
        g_iso.replay()
        i0 = torch.cuda.Event(enable_timing=True)
        i1 = torch.cuda.Event(enable_timing=True)
        i0.record(stream)
        for _ in range(max(1, iso_steps // min(G, iso_steps))):
            g_iso.replay()
        i1.record(stream)
    stream.synchronize()
    iso_plan = ctx.last_plan()
    # End to end the inputs arrive by host copies on the same stream, which the
    # library does not track: the library's default (no early start).
    iso_s = i0.elapsed_time(i1) / 1e3 / (max(1, iso_steps // min(G, iso_steps)) * min(G, iso_steps))

    unit_bytes = layer.algorithmic_bytes()
    max_s, total_units = aggregate(local_s, float(steps) * unit_bytes, world, dev)
    per_launch_s = local_s / steps
    hbm_bound = unit_bytes / 6.8e12 >= layer.flops / 1.9e15 if layer.precision != si.PREC_FP32 else False
    if hbm_bound:
        value, unit = total_units / max_s / 1e9, "GB/s"
    else:
        value, unit = world * steps * layer.flops / max_s / 1e12, "TFLOP/s"

    peaks, src = load_peaks()
    kfile = {tll.KERNEL_SKINNY: "skinny.cu", tll.KERNEL_FFMA: "ffma.cu", tll.KERNEL_TC: "tc.cu",
             tll.KERNEL_GEMV: "gemv.cu"}.get(plan.kernel)
    traffic = traffic_from_profile(kfile, layer.name) if kfile else None
    roof = roofline_for(layer, per_launch_s, peaks, src, traffic)

    # End to end through the public API with host buffers: pinned host X, W,
    # bias in, Y out, every step, copies inside the timed region.
    hx = torch.from_numpy(X).to(dt).pin_memory()
    hw = torch.from_numpy(W).to(dt).pin_memory()
    hb = None if b is None else torch.from_numpy(b).pin_memory()
    hy = torch.empty((layer.M, layer.N), dtype=dt).pin_memory()
    dx, dw = torch.empty_like(x), torch.empty_like(w0)
    db = None if bias is None else torch.empty_like(bias)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        if db is not None:
            db.copy_(hb, non_blocking=True)
        out = tll.forward(dx, dw, db, epilogue=epi, precision=prec, ctx=ctx)
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
    h2d = hx.numel() * esz + hw.numel() * esz + (0 if hb is None else hb.numel() * 4)
    d2h = hy.numel() * esz
    e2e_val = unit_bytes / e2e_s / 1e9 if unit == "GB/s" else layer.flops / e2e_s / 1e12
    e2e = {"value": round(e2e_val * world, 3), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": e2e_steps, "api": "transformer_linear_layer_gb300.forward (C ABI lin_forward)"}
    iso_val = unit_bytes / iso_s / 1e9 if unit == "GB/s" else layer.flops / iso_s / 1e12
    isolated = {"value": round(iso_val, 3), "unit": unit, "ms_per_step": round(iso_s * 1e3, 6),
                "plan": {k: v for k, v in iso_plan.as_dict().items() if k != "kernel_name"},
                "note": "early start off (the library default): each call waits for the previous kernel"}

    cpu = None
    if with_cpu_baseline and rank == 0:
        cpu = cpu_baseline(layer, X, W, b, unit)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(max_s / steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": prec, "data": "synthetic",
        "config": {"workload": layer.name, "M": layer.M, "N": layer.N, "K": layer.K,
                   "bias": layer.bias, "epilogue": epi, "precision": prec,
                   "kernel": plan.as_dict()["kernel_name"],
                   "plan": {k: v for k, v in plan.as_dict().items() if k != "kernel_name"},
                   "l2": f"cold W: {n_copies} rotating copies of W ({n_copies * w_bytes >> 20} MiB > L2 "
                         f"{l2 >> 20} MiB), steps replayed from a CUDA graph of {G}",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "parity_gate": {"rel_err": err, "rel_err_after_timed_steps": err_after, "tol": tol,
                                   "compared": gate},
                   "steps_are": "independent back-to-back calls (same X, rotating W copies) with the early "
                                "start at level 2 (LIN_OPT_EARLY_START): a call may start and read its inputs "
                                "before its predecessor finishes and writes Y after it; e2e and isolated_call "
                                "use the library default (off)"},
        "isolated_call": isolated,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": steps * (0 if plan.kernel in (tll.KERNEL_NONE,) else 1),
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
    rotating over copies larger than L2, replayed from a CUDA graph; parity
    gate on sampled output rows against the oracle."""
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
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.integers(0, out.shape[0], 64), [0, out.shape[0] - 1]]))
    if work.which == 1:
        ref = oracle.backward_dx(dZ[rows], B)
    elif work.which == 2:
        ref, _ = oracle.backward_dw(dZ[:, rows], B, with_bias=False)
    elif work.which == 3:
        ref = oracle.backward_dx_gelu(dZ[rows], B, Zp[rows])
    else:
        ref = oracle.linear_residual(dZ[rows], B, R[rows], bias_h)
    got = out[torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    err = oracle.rel_err(got, ref)
    tol = oracle.TOL[si.PREC_BF16] if work.precision == si.PREC_BF16 else oracle.TOL[si.PREC_FP32]
    if not err <= tol:
        raise SystemExit(f"correctness gate failed for {work.name}: rel_err {err} > {tol}")

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    stream.synchronize()
    G = n_copies * max(1, 64 // n_copies)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                step(i)
        return g

    graph = capture(G)
    rem = steps % G
    graph_rem = capture(rem) if rem else None
    stream.synchronize()
    sampler = ClockSampler(local_rank)
    soak_until = time.perf_counter() + 1.0
    with torch.cuda.stream(stream):
        while time.perf_counter() < soak_until:
            graph.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // G):
            graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
        e1.record(stream)
    stream.synchronize()
    barrier(world)
    clocks = sampler.stop()
    local_s = e0.elapsed_time(e1) / 1e3
    ctx.check(stream)
    got = out[torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    err_after = oracle.rel_err(got, ref)
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
                         f"({n_copies * rot_bytes >> 20} MiB > L2 {l2 >> 20} MiB), "
                         f"steps replayed from a CUDA graph of {G}",
                   "parity_gate": {"rel_err": err, "rel_err_after_timed_steps": err_after, "tol": tol,
                                   "compared": f"{len(rows)} sampled output rows"}},
        "roofline": roof, "clocks": clocks, "gpu_launches": steps,
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
    hbm_bound = layer.precision != si.PREC_FP32 and layer.algorithmic_bytes() / 6.8e12 >= layer.flops / 1.9e15
    unit = "GB/s" if hbm_bound else "TFLOP/s"
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


# ------------------------------------------------------------------- main

BWD_BY_NAME = {w.name: w for w in BWD_WORKLOADS}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(BWD_BY_NAME))
    ap.add_argument("--all", action="store_true", help="one line per workload (stdout), default line last")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    steps, warmup = max(1, args.steps), max(3, args.warmup)

    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.workload in BWD_BY_NAME:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times forward workloads only"}))
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

    if args.workload in BWD_BY_NAME:
        work = BWD_BY_NAME[args.workload]
        line = bench_backward(work, steps, warmup, world, rank, local_rank)
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
    for name in names:
        layer = WORKLOADS[name]
        # Other workloads: at least 300 steps and ~20 TFLOP, so that the timed
        # region spans several replays of the step graph.
        st = steps if name == args.workload else max(300, min(steps, int(2e13 / max(layer.flops, 1e6))))
        line = bench_ours(layer, st, warmup, world, rank, local_rank,
                          with_cpu_baseline=(not args.no_cpu_baseline and name == args.workload),
                          e2e_steps=args.e2e_steps if name == args.workload else 5)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
