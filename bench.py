"""Benchmark of the fused NHWC convolution layer on GB300.

One step = one pass of every layer of the batch-8 bf16 throughput sweep
(3x3 64->128 @160x160, 3x3 256->256 @80x80, 3x3 512->1024 @40x40,
1x1 1024->512 @20x20, depthwise 3x3 512 @40x40; Mish epilogue), inputs
resident in HBM, through the library's C ABI.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Timing: one step (the five conv_run calls, with a CUDA event before each and
one after the last) is captured once as a CUDA graph; W untimed warm-up
replays, then K timed replays.  Before every replay the L2 is flushed (a
write of a buffer twice the L2 size) outside the step's events.  The events
inside the graph give the per-layer durations and the dominant kernel's
roofline, without host launch gaps between layers.  `value` = algorithmic FLOPs (2 * MACs) of all layers of all ranks
/ the slowest rank's summed step time.  `e2e` times the same step through
the same API from pinned host buffers (host->device copies of x, w, b and
device->host copy of y inside the timed region).  `cpu_baseline` times the
CPU oracle on a bounded random sample of output points of the same layers.
`--impl reference` times that oracle alone on the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused conv TFLOP/s (bf16) & TOPS (int8) per layer shape; % of GB300 roofline"
DEFAULT_WORKLOAD = "sweep_b8_bf16"
# Fallback peaks (one earlier GB300 measurement) when MEASURED_PEAKS.json is absent.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def flops_of(spec):
    from conv_workloads import macs
    return 2.0 * macs(spec)


def compute_peak(spec, peaks):
    """The compute roof of a layer's own arithmetic: bf16 layers and the int8
    layers (which this library contracts as exact bf16 MMAs) take the measured
    bf16 tensor peak; fp32 layers (FFMA, never TF32) the FFMA peak, SMs x 128
    lanes x 2 flops x the maximum SM clock.  Returns (TFLOP/s, roof name)."""
    if spec.dtype == "f32":
        return peaks["fp32_ffma_tflops"], "alu"
    return peaks["bf16_tflops"], "tensor"


def layer_bound(spec, peaks):
    """Which roof binds a layer: compare its arithmetic intensity with the
    ridge (its compute peak / HBM bandwidth)."""
    from conv_workloads import alg_bytes
    ai = flops_of(spec) / alg_bytes(spec)
    pk, roof = compute_peak(spec, peaks)
    ridge = pk * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return (roof if ai >= ridge else "hbm"), ai


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons every 50 ms while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self, window_s=None):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # samples of the main timed region (+ one sampling period), and of
        # every GPU timing phase up to t_last
        t0, t1 = getattr(self, "t_start", 0.0), getattr(self, "t_end", 1e30) + 0.06
        n_main = sum(1 for ts, _ in self.lines if t0 <= ts <= t1)
        t_last = getattr(self, "t_last", 1e30) + 0.06
        inside = [ln for ts, ln in self.lines if ts <= t_last]
        where = ("warm-up, the timed step replays and every later GPU timing phase (per-layer, other "
                 "layer sets, adjacent rows)")
        if window_s is not None:
            where += f": {window_s:.1f} s"
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "sm_min_mhz": min(sm),
                "reasons": sorted(reasons), "samples": len(sm), "samples_in_step_region": n_main,
                "window": where}


# ---------------------------------------------------------------- replicas

def max_over_ranks(ms, world, device):
    """The slowest rank's time: every rank runs the same fixed work (weak
    scaling, no data-path collective), so the job takes as long as its
    slowest replica.  `device` is where the reduction runs (the rank's GPU
    under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, world, steps, ms):
    """Whole-job throughput: the work of every rank's `steps` steps over the
    slowest rank's time (ms)."""
    return flops_per_step * world * steps / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- per-layer timing

class GraphTimer:
    """CUDA-graph timing helpers on one device, with an L2-flush buffer."""

    def __init__(self, dev, flush):
        self.dev, self.flush = dev, flush

    def capture(self, fn, with_events=False):
        """fn captured as a CUDA graph (optionally between two timing events,
        external=True so each replay re-records them)."""
        import torch
        evs = None
        if with_events:
            evs = (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = torch.cuda.current_stream(self.dev)
            if evs:
                evs[0].record(st)
            fn()
            if evs:
                evs[1].record(st)
        return g, evs

    def graph_us(self, fn, reps=5):
        """Best of `reps` replays of fn captured between two events, in us."""
        import torch
        g, (ea, eb) = self.capture(fn, with_events=True)
        best = None
        for _ in range(reps):
            g.replay()
            torch.cuda.synchronize()
            t = ea.elapsed_time(eb) * 1e3
            best = t if best is None else min(best, t)
        del g
        return best

    def launch_floor(self, cl, R=20):
        """A layer of almost no work (depthwise 3x3 on one 8x8x8 bf16 image)
        R times back to back in one graph, per launch."""
        import torch
        tiny = cl.Plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 8, "bf16", "none")
        tx = torch.zeros(1, 8, 8, 8, dtype=torch.bfloat16, device=self.dev)
        tw = torch.zeros(8, 3, 3, 1, dtype=torch.bfloat16, device=self.dev)
        ty = torch.empty(1, 8, 8, 8, dtype=torch.bfloat16, device=self.dev)

        def tiny_run():
            st = torch.cuda.current_stream(self.dev)
            for _ in range(R):
                tiny.run(tx, tw, None, ty, st)
        tiny_run()
        torch.cuda.synchronize()
        return self.graph_us(tiny_run) / R


def measure_set(tm, plans, X, Wt, B, Y, pairs=50, R=20):
    """Per-layer times of one layer set on the GPU, in us:
      marginal_us  the layer's cost inside the step: the step's graph (the
                   layers back to back, programmatic dependent launch between
                   them) minus the same graph without that layer, each replay
                   after an L2 flush, interleaved, mean of `pairs` replays (a
                   set of one layer: the graph of the layer twice minus the
                   graph of it once);
      evented_us   events recorded between consecutive layers of the step
                   (they serialise the layers: reads high by the event cost);
      cold_us / warm_us  the layer alone, R launches in one graph, cold as
                   [flush, layer] x R minus [flush] x R, warm back to back,
                   divided by R;
      step_us      the whole step (mean of the same replays)."""
    import torch
    dev, flush = tm.dev, tm.flush
    nl = len(plans)

    def step_without(skip):
        def f():
            st = torch.cuda.current_stream(dev)
            for i in range(nl):
                if i != skip:
                    plans[i].run(X[i], Wt[i], B[i], Y[i], st)
        return f

    def twice():  # (a set of one layer: the graph of the layer run twice)
        st = torch.cuda.current_stream(dev)
        for _ in range(2):
            plans[0].run(X[0], Wt[0], B[0], Y[0], st)

    stream = torch.cuda.current_stream(dev)
    step_without(None)()
    torch.cuda.synchronize()
    graphs = [tm.capture(step_without(None))[0]]
    if nl > 1:
        graphs += [tm.capture(step_without(i))[0] for i in range(nl)]
    else:
        graphs.append(tm.capture(twice)[0])
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in graphs]
          for _ in range(pairs)]
    for k in range(pairs):
        for j, g in enumerate(graphs):
            flush.fill_((k + j) & 0xFF)
            ev[k][j][0].record(stream)
            g.replay()
            ev[k][j][1].record(stream)
    torch.cuda.synchronize()
    t = np.array([[a.elapsed_time(b) * 1e3 for a, b in row] for row in ev])
    del graphs
    step_us = float(t[:, 0].mean())
    # a layer's cost in the step; for a set of one layer, what a second copy
    # of it adds to the graph (the graph's own launch cost is not the layer's)
    marginal = ([float(t[:, 1].mean()) - step_us] if nl == 1
                else [step_us - float(t[:, 1 + i].mean()) for i in range(nl)])

    # events between the layers
    lev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nl + 1)]

    def evented_step():
        st = torch.cuda.current_stream(dev)
        for i in range(nl):
            lev[i].record(st)
            plans[i].run(X[i], Wt[i], B[i], Y[i], st)
        lev[nl].record(st)
    gl, _ = tm.capture(evented_step)
    reps = 10
    ev_us = np.zeros((reps, nl))
    for k in range(reps):
        flush.fill_(k & 0xFF)
        gl.replay()
        torch.cuda.synchronize()
        for i in range(nl):
            ev_us[k, i] = lev[i].elapsed_time(lev[i + 1]) * 1e3
    del gl

    def flushes():
        for r in range(R):
            flush.fill_(r & 0xFF)
    t_flush = tm.graph_us(flushes)
    cold, warm = [], []
    for i in range(nl):
        def c(i=i):
            st = torch.cuda.current_stream(dev)
            for r in range(R):
                flush.fill_(r & 0xFF)
                plans[i].run(X[i], Wt[i], B[i], Y[i], st)

        def w(i=i):
            st = torch.cuda.current_stream(dev)
            for _ in range(R):
                plans[i].run(X[i], Wt[i], B[i], Y[i], st)
        cold.append((tm.graph_us(c) - t_flush) / R)
        warm.append(tm.graph_us(w) / R)
    return {"step_us": step_us, "marginal_us": marginal, "evented_us": list(ev_us.mean(axis=0)),
            "cold_us": cold, "warm_us": warm}


def rate_of(spec, us, peaks):
    """(achieved, peak, unit, bound) of a layer that took `us`: against its
    compute roof (TFLOP/s, TOPS for int8, FFMA TFLOP/s for fp32) or HBM
    (GB/s), whichever its arithmetic intensity puts it under."""
    from conv_workloads import alg_bytes
    bound, _ = layer_bound(spec, peaks)
    if bound != "hbm":
        unit = "TOPS" if spec.dtype == "i8" else "TFLOP/s"
        return flops_of(spec) / (us * 1e-6) / 1e12, compute_peak(spec, peaks)[0], unit, bound
    return alg_bytes(spec) / (us * 1e-6) / 1e9, peaks["hbm_gbs"], "GB/s", bound


def layer_row(spec, plan, meas, i, peaks):
    from conv_workloads import alg_bytes
    us = max(float(meas["marginal_us"][i]), 1e-3)
    cold = float(meas["cold_us"][i])
    ach, pk, unit, bound = rate_of(spec, us, peaks)
    ach_c = rate_of(spec, cold, peaks)[0]
    _, ai = layer_bound(spec, peaks)
    ops = "tops" if spec.dtype == "i8" else "tflops"
    return {
        "layer": spec.name, "kernel": plan.describe(), "launches": plan.launches, "us": round(us, 2),
        "us_evented": round(float(meas["evented_us"][i]), 2),
        "us_alone_cold": round(cold, 2), "us_alone_warm": round(float(meas["warm_us"][i]), 2),
        ops: round(flops_of(spec) / (us * 1e-6) / 1e12, 2), "gbs": round(alg_bytes(spec) / (us * 1e-6) / 1e9, 1),
        "ai_flop_per_byte": round(ai, 1), "bound": bound,
        "achieved": round(ach, 2), "peak": pk, "unit": unit, "frac": round(ach / pk, 4),
        "frac_alone_cold": round(ach_c / pk, 4),
    }


def measure_layer_set(cl, dev, tm, cfg, peaks):
    """One of the other layer sets, each layer planned as a user would plan
    it, timed as the main set's layers are (measure_set)."""
    import torch
    from conv_workloads import generate
    layers = generate(cfg)
    plans, X, Wt, B, Y = [], [], [], [], []
    for d in layers:
        s = d.spec
        quant = (s.in_scale, s.out_scale, d.w_scales.tolist()) if s.dtype == "i8" else None
        p = cl.Plan(s.n, s.h, s.w, s.cin, s.cout, s.kh, s.kw, s.stride, s.pad_h, s.pad_w, s.groups,
                    s.dtype, s.act, quant)
        plans.append(p)
        X.append(d.x.to(dev))
        Wt.append(d.w.to(dev))
        B.append(None if d.b is None else d.b.to(dev))
        Y.append(torch.empty(p.output_shape, dtype=d.x.dtype, device=dev))
    meas = measure_set(tm, plans, X, Wt, B, Y)
    rows = [layer_row(d.spec, p, meas, i, peaks) for i, (d, p) in enumerate(zip(layers, plans))]
    for p in plans:
        p.check_device_status()
    flops = sum(flops_of(d.spec) for d in layers)
    ops = "TOPS" if all(d.spec.dtype == "i8" for d in layers) else "TFLOP/s"
    return {"step_us": round(meas["step_us"], 2), "rate": round(flops / (meas["step_us"] * 1e-6) / 1e12, 3),
            "unit": ops, "layers": rows}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, device):
    import torch

    import convolution_nhwc_implicit_gb300 as cl
    from conv_workloads import CONFIGS, alg_bytes, generate, macs, output_hw

    peaks, peaks_src = load_peaks()
    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    # FFMA peak of the fp32 layers: SMs x 128 FP32 lanes x 2 flops x max SM clock
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    peaks["fp32_ffma_tflops"] = round(props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12, 1)
    layers = generate(args.workload)
    if args.only:  # (profile pass) just these layers of the set
        layers = [d for d in layers if d.spec.name in args.only.split(",")]
        if not layers:
            raise SystemExit(f"--only: no layer of {args.workload} is named {args.only}")
    plans, X, Wt, B, Y = [], [], [], [], []
    for d in layers:
        s = d.spec
        quant = (s.in_scale, s.out_scale, d.w_scales.tolist()) if s.dtype == "i8" else None
        p = cl.Plan(s.n, s.h, s.w, s.cin, s.cout, s.kh, s.kw, s.stride, s.pad_h, s.pad_w, s.groups,
                    s.dtype, s.act, quant)
        plans.append(p)
        X.append(d.x.to(dev))
        Wt.append(d.w.to(dev))
        B.append(None if d.b is None else d.b.to(dev))
        Y.append(torch.empty(p.output_shape, dtype=d.x.dtype, device=dev))
    stream = torch.cuda.current_stream(dev)
    if args.profile_pass:
        # For a profiler's launch list: `warmup` eager passes over the layers,
        # then one more, each layer's launches in order, no graphs, no timing.
        for _ in range(args.warmup + 1):
            for i in range(len(layers)):
                plans[i].run(X[i], Wt[i], B[i], Y[i], stream)
        torch.cuda.synchronize()
        return {"profile_pass": args.workload, "passes": args.warmup + 1,
                "launches_per_pass": sum(p.launches for p in plans),
                "layers": [{"layer": d.spec.name, "kernel": p.describe(), "launches": p.launches}
                           for d, p in zip(layers, plans)]}
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    nl = len(layers)
    tm = GraphTimer(dev, flush)

    def step():
        st = torch.cuda.current_stream(dev)  # the capture stream while capturing
        for i in range(nl):
            plans[i].run(X[i], Wt[i], B[i], Y[i], st)

    # The step (the layers back to back, nothing between them: consecutive
    # launches overlap through programmatic dependent launch) is captured as
    # one CUDA graph and replayed, so the GPU never waits on the host.
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    graph, _ = tm.capture(step)
    torch.cuda.synchronize()

    # Clocks are sampled from the first warm-up replay to the end of the last
    # timed phase (the step, the per-layer figures, the other layer sets and
    # the adjacent rows): the step's own timed region is a few milliseconds,
    # shorter than the sampling period.
    clocks = ClockSampler(device)
    clocks.start()
    t_sampling = time.perf_counter()
    for _ in range(args.warmup):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks.mark("t_start")
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)          # outside the events: L2 holds none of the step's inputs
        e0[k].record(stream)
        graph.replay()
        e1[k].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks.mark("t_end")
    step_ms = np.array([e0[k].elapsed_time(e1[k]) for k in range(args.steps)])
    del graph

    meas = measure_set(tm, plans, X, Wt, B, Y)
    layer_rows = [layer_row(d.spec, p, meas, i, peaks) for i, (d, p) in enumerate(zip(layers, plans))]
    launch_floor = tm.launch_floor(cl)
    for p in plans:
        p.check_device_status()
    my_ms = max_over_ranks(float(step_ms.sum()), world, dev)
    total_flops = sum(flops_of(d.spec) for d in layers)
    ms_per_step = my_ms / args.steps
    value = job_tflops(total_flops, world, args.steps, my_ms)

    # ---- the dominant kernel's roofline: the layer taking the most time in
    # the step (its marginal time there: the step minus the step without it)
    dom = max(range(nl), key=lambda i: meas["marginal_us"][i])
    dr = layer_rows[dom]
    traffic = _traffic_for(args.workload, layers[dom].spec.name, plans[dom].describe())
    roofline = {"bound": dr["bound"], "achieved": dr["achieved"], "peak": dr["peak"], "unit": dr["unit"],
                "frac": dr["frac"], "traffic": traffic, "kernel": layers[dom].spec.name,
                "duration_us": dr["us"], "duration": "marginal time in the step (CUDA events)",
                "peak_source": {"tensor": f"{peaks_src} (bf16 burst)", "hbm": f"{peaks_src} (HBM copy)",
                                "alu": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}[dr["bound"]]}

    # ---- the other layer sets, each measured the same way (rank 0 only)
    layer_sets = None
    if rank == 0 and not args.only and not args.no_layer_sets:
        layer_sets = {}
        for cfg in CONFIGS:
            if cfg == args.workload:
                continue
            layer_sets[cfg] = measure_layer_set(cl, dev, tm, cfg, peaks)

    # ---- int8 context: the tensor cores' int8 rate as torch exposes it (these
    # layers themselves run as exact bf16 MMAs, so their roof is the bf16 peak)
    int8_probe = None
    if any(d.spec.dtype == "i8" for d in layers) or "vww_int8" in (layer_sets or {}):
        try:
            a8 = torch.randint(-128, 128, (8192, 8192), dtype=torch.int8, device=dev)
            b8 = torch.randint(-128, 128, (8192, 8192), dtype=torch.int8, device=dev).t()
            best = None
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch._int_mm(a8, b8)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
            int8_probe = {"int8_tops": round(2 * 8192 ** 3 / (best * 1e-3) / 1e12, 1),
                          "how": "torch._int_mm 8192^3, best of 10"}
            del a8, b8
        except Exception as e:  # no int8 GEMM in this torch build
            int8_probe = {"unavailable": str(e)[:120]}

    # ---- end to end through the same API, from pinned host memory
    e2e = run_e2e(args, layers, plans, dev, stream, total_flops, world)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "layers": len(layers),
                   "batch_per_gpu": layers[0].spec.n, "l2": "flushed before every step (outside the events)",
                   "launch": "CUDA graph replay of the step, events around each replay; per-layer 'us': "
                             "the layer's marginal time in the step (the step graph minus the same graph "
                             "without that layer, L2 flushed before each replay, mean of 50 pairs); "
                             "'us_evented': events between the layers; 'us_alone_*': each layer 20x in its "
                             "own graph",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline, "layers": layer_rows, "e2e": e2e,
        "peaks": {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"],
                  "fp32_ffma_tflops": peaks["fp32_ffma_tflops"], "source": peaks_src,
                  "int8_probe": int8_probe},
        "layer_sets": layer_sets,
        "next_rows": measure_next_rows(dev, peaks) if rank == 0 and not args.no_next_rows else None,
        "launch_floor_us": round(float(launch_floor), 2),
        "gpu_launches": sum(p.launches for p in plans) * args.steps,
        "wall_s_timed_region": round(wall, 4),
    }
    torch.cuda.synchronize()
    clocks.mark("t_last")
    out["clocks"] = clocks.stop(time.perf_counter() - t_sampling)
    return out


def measure_next_rows(dev, peaks, reps=20):
    """The adjacent rows built beyond the five layer sets (the residual-add
    epilogue, concat + 2x upsample output placement, the SPP block, the fused
    depthwise -> pointwise pair), each timed like a layer alone in the main
    step: `reps` calls, each after an L2 flush, captured in one CUDA graph
    between two events, minus the same graph of flushes alone, divided by
    `reps`; reported with its roofline."""
    import torch
    import convolution_nhwc_implicit_gb300 as cl
    from conv_workloads import LayerSpec, alg_bytes, make_layer

    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def graph_us(body):
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = torch.cuda.current_stream(dev)
            e0.record(st)
            body()
            e1.record(st)
        best = None
        for _ in range(5):
            g.replay()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e3
            best = t if best is None else min(best, t)
        del g
        return best

    def flushes():
        for r in range(reps):
            flush.fill_(r & 0xFF)

    t_flush = graph_us(flushes)

    def timed(fn):
        fn()
        torch.cuda.synchronize()

        def body():
            for r in range(reps):
                flush.fill_(r & 0xFF)
                fn()
        return (graph_us(body) - t_flush) / reps

    def roof(flops, nbytes, us):
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        if flops / nbytes >= ridge:
            a = flops / (us * 1e-6) / 1e12
            return {"bound": "tensor", "achieved": round(a, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(a / peaks["bf16_tflops"], 4)}
        a = nbytes / (us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(a, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(a / peaks["hbm_gbs"], 4)}

    rows = []
    g = torch.Generator("cpu").manual_seed(5)
    # 1. residual add: the batch-8 256->256 3x3 layer with a skip tensor
    s = LayerSpec("conv3x3_256to256_80_residual", 8, 80, 80, 256, 256, 3, 3, 1, 1, 1, dtype="bf16",
                  act="mish", x_dist=("normal", 1.0))
    d = make_layer(s, g)
    x, w, b = d.x.to(dev), d.w.to(dev), d.b.to(dev)
    r = torch.randn(8, 80, 80, 256, generator=g).to(torch.bfloat16).to(dev)
    y = torch.empty(8, 80, 80, 256, dtype=torch.bfloat16, device=dev)
    pf = cl.Plan(8, 80, 80, 256, 256, 3, 3, 1, 1, 1, 1, "bf16", "mish", out=dict(residual=True))
    pp = cl.Plan(8, 80, 80, 256, 256, 3, 3, 1, 1, 1, 1, "bf16", "mish")
    us = timed(lambda: pf.run(x, w, b, y, residual=r))
    us_plain = timed(lambda: pp.run(x, w, b, y))
    rows.append(dict({"row": "residual add (K2)", "layer": s.name, "kernel": pf.describe(), "us": round(us, 2),
                      "plain_us": round(us_plain, 2)},
                     **roof(flops_of(s), alg_bytes(s) + r.numel() * 2, us)))
    # 2. concat + 2x upsample: YOLOv4 neck 1x1 512->256 at 20x20 (batch 8) written
    #    upsampled into channels 256..511 of a 40x40x512 concat buffer
    s = LayerSpec("pw1x1_512to256_20_up2_concat", 8, 20, 20, 512, 256, 1, 1, dtype="bf16", act="mish",
                  x_dist=("normal", 1.0))
    d = make_layer(s, g)
    x, w, b = d.x.to(dev), d.w.to(dev), d.b.to(dev)
    ycat = torch.empty(8, 40, 40, 512, dtype=torch.bfloat16, device=dev)
    pc = cl.Plan(8, 20, 20, 512, 256, 1, 1, 1, 0, 0, 1, "bf16", "mish",
                 out=dict(y_channels=512, y_channel_offset=256, upsample=2))
    us = timed(lambda: pc.run(x, w, b, ycat))
    nbytes = alg_bytes(s) + 3 * 8 * 20 * 20 * 256 * 2  # the output is written four times
    rows.append(dict({"row": "concat + 2x upsample (K4)", "layer": s.name, "kernel": pc.describe(),
                      "us": round(us, 2)}, **roof(flops_of(s), nbytes, us)))
    # 3. SPP: 8 x 20 x 20 x 512 bf16 -> [mp5 | mp9 | mp13 | x] (2048 channels)
    xs = torch.randn(8, 20, 20, 512, generator=g).to(torch.bfloat16).to(dev)
    ys = torch.empty(8, 20, 20, 2048, dtype=torch.bfloat16, device=dev)
    us = timed(lambda: cl.spp(xs, ys))
    nbytes = xs.numel() * 2 + ys.numel() * 2
    rows.append(dict({"row": "SPP max pools 5/9/13 (K3)", "layer": "spp_20x20x512_b8", "kernel": "spp cascaded 5x5",
                      "us": round(us, 2)}, **roof(0.0, nbytes, us)))
    # 4. fused depthwise -> pointwise pair: the KWS DS-CNN block (1x25x5x64,
    #    fp32, ReLU / ReLU), beside the same two layers run as two plans
    xk = torch.empty(1, 25, 5, 64).uniform_(-1, 1, generator=g).to(dev)
    wd = (torch.randn(64, 3, 3, 1, generator=g) * (2 / 9) ** 0.5).to(dev)
    bd = (torch.randn(64, generator=g) * 0.01).to(dev)
    wp = (torch.randn(64, 1, 1, 64, generator=g) * (2 / 64) ** 0.5).to(dev)
    bp = (torch.randn(64, generator=g) * 0.01).to(dev)
    yk = torch.empty(1, 25, 5, 64, device=dev)
    zk = torch.empty(1, 25, 5, 64, device=dev)
    pf = cl.DwpwPlan(1, 25, 5, 64, 64, 1, 1, "f32", "relu", "relu")
    p1 = cl.Plan(1, 25, 5, 64, 64, 3, 3, 1, 1, 1, 64, "f32", "relu")
    p2 = cl.Plan(1, 25, 5, 64, 64, 1, 1, 1, 0, 0, 1, "f32", "relu")
    us = timed(lambda: pf.run(xk, wd, bd, wp, bp, yk))

    def two():
        p1.run(xk, wd, bd, zk)
        p2.run(zk, wp, bp, yk)
    us_two = timed(two)
    fl = 2.0 * 125 * 64 * (9 + 64)
    nbytes = 4 * (125 * 64 * 2 + 64 * 9 + 64 * 64 + 128)
    ach = nbytes / (us * 1e-6) / 1e9  # far below the FFMA ridge: HBM (latency) bound
    rows.append({"row": "fused dw3x3 -> pw1x1 (DS-CNN block)", "layer": "kws_ds_block_25x5x64_f32",
                 "kernel": pf.describe(), "us": round(us, 2), "plain_us": round(us_two, 2),
                 "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": round(ach / peaks["hbm_gbs"], 4),
                 "tflops": round(fl / (us * 1e-6) / 1e12, 3),
                 "note": "plain_us: the depthwise and pointwise plans run one after the other"})
    return rows


def run_e2e(args, layers, plans, dev, stream, total_flops, world):
    """Same step, but inputs start in pinned host memory and y returns to it.

    Pipelined over three streams, as a serving loop would run it: uploads of
    x, w, b on one, the layers on the compute stream, downloads of y on a
    third, each layer waiting for its own upload and each download for its
    own layer; two sets of device buffers let step k + 1's uploads run while
    step k computes and downloads.  Every step still copies all its inputs
    in and all its outputs out inside the timed region."""
    import torch
    hx = [d.x.pin_memory() for d in layers]
    hw = [d.w.pin_memory() for d in layers]
    hb = [None if d.b is None else d.b.pin_memory() for d in layers]
    hy = [[torch.empty(p.output_shape, dtype=d.x.dtype).pin_memory() for p, d in zip(plans, layers)]
          for _ in range(2)]
    nb = 2  # device buffer sets
    dx = [[torch.empty_like(t, device=dev) for t in hx] for _ in range(nb)]
    dw = [[torch.empty_like(t, device=dev) for t in hw] for _ in range(nb)]
    db = [[None if t is None else torch.empty_like(t, device=dev) for t in hb] for _ in range(nb)]
    dy = [[torch.empty(t.shape, dtype=t.dtype, device=dev) for t in hy[0]] for _ in range(nb)]
    h2d = sum(t.numel() * t.element_size() for t in hx + hw + [t for t in hb if t is not None])
    d2h = sum(t.numel() * t.element_size() for t in hy[0])
    s_up = torch.cuda.Stream(dev)
    s_down = torch.cuda.Stream(dev)
    nl = len(plans)
    ev = lambda: torch.cuda.Event()  # noqa: E731 (synchronisation only)
    up_done = [[ev() for _ in range(nl)] for _ in range(nb)]
    run_done = [[ev() for _ in range(nl)] for _ in range(nb)]
    down_done = [[ev() for _ in range(nl)] for _ in range(nb)]
    started = [[False] * nl for _ in range(nb)]

    def step(k):
        j = k % nb
        for i, p in enumerate(plans):
            with torch.cuda.stream(s_up):
                if started[j][i]:
                    s_up.wait_event(run_done[j][i])  # the layer that last read these inputs is done
                dx[j][i].copy_(hx[i], non_blocking=True)
                dw[j][i].copy_(hw[i], non_blocking=True)
                if hb[i] is not None:
                    db[j][i].copy_(hb[i], non_blocking=True)
                up_done[j][i].record(s_up)
            stream.wait_event(up_done[j][i])
            if started[j][i]:
                stream.wait_event(down_done[j][i])  # y of this buffer set has been read back
            p.run(dx[j][i], dw[j][i], db[j][i], dy[j][i], stream)
            run_done[j][i].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(run_done[j][i])
                hy[j][i].copy_(dy[j][i], non_blocking=True)
                down_done[j][i].record(s_down)
            started[j][i] = True

    for k in range(max(1, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    k = max(1, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for i in range(k):
        step(i)
    e1.record(s_down)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    return {"value": round(job_tflops(total_flops, world, k, ms), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / k, 4),
            "how": "uploads, layers and downloads on three streams, two device buffer sets"}


# Source files that define each kernel family (a change to any of them voids
# the DRAM traffic captured for that family).
_FAMILY_SOURCES = {
    "igemm": ["k_igemm.cu", "k_igemm_ept.cu", "k_igemm_cvt.cu", "k_igemm_kernel.cuh", "k_prep.cu", "tc_ptx.cuh", "epilogue.cuh",
              "conv_internal.h"],
    "dw3x3+pw1x1": ["k_dwpw.cu", "epilogue.cuh", "conv_internal.h"],
    "dw3x3": ["k_dw3x3.cu", "tc_ptx.cuh", "epilogue.cuh", "conv_internal.h"],
    "direct": ["k_direct.cu", "epilogue.cuh", "conv_internal.h"],
}


def kernel_sources_sha1(kernel_desc):
    """sha1 of the source files of the kernel family a plan description names."""
    import hashlib
    fam = next((f for f in _FAMILY_SOURCES if kernel_desc.startswith(f)), None)
    if fam is None:
        return None
    h = hashlib.sha1()
    for name in _FAMILY_SOURCES[fam]:
        with open(os.path.join(ROOT, "convolution_nhwc_implicit_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def _traffic_for(workload, layer_name, kernel_desc):
    """DRAM bytes per launch of this kernel from the committed ncu summary
    (profiles/dram_traffic.json), if it was captured for this exact kernel
    configuration and its sources have not changed since; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(layer_name)
    if not e or e.get("kernel") != kernel_desc or e.get("sources_sha1") != kernel_sources_sha1(kernel_desc):
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(layers, budget_s, seed=0):
    """Times the oracle on a bounded random sample of output points of every
    layer, sized from a short calibration so the whole sample takes about
    budget_s seconds.  Returns (flops_done, seconds, points, threads)."""
    import oracle
    from conv_workloads import macs, output_hw
    prepared = []
    for d in layers:
        s = d.spec
        if s.dtype == "i8":
            M = oracle.requant_multipliers(s.in_scale, s.out_scale, d.w_scales.numpy())
            prepared.append((s, d.x.numpy(), d.w.numpy(), None if d.b is None else d.b.numpy(), M))
        else:
            prepared.append((s, d.x.double().numpy(), d.w.double().numpy(),
                             None if d.b is None else d.b.double().numpy(), None))
    rng = np.random.default_rng(seed)

    def pts_for(s, count):
        oh, ow = output_hw(s)
        return np.stack([rng.integers(0, s.n, count), rng.integers(0, oh, count), rng.integers(0, ow, count),
                         rng.integers(0, s.cout, count)], axis=1).astype(np.int32)

    def run(frac):
        fl, secs, npts = 0.0, 0.0, 0
        for s, x, w, b, M in prepared:
            oh, ow = output_hw(s)
            total = s.n * oh * ow * s.cout
            count = max(16, int(total * frac))
            pts = pts_for(s, count)
            t0 = time.perf_counter()
            if M is not None:
                oracle.conv_i8_points(x, w, b, M, pts, s.stride, s.pad_h, s.pad_w, s.groups, s.act == "relu")
            else:
                oracle.conv_f64_points(x, w, b, pts, s.stride, s.pad_h, s.pad_w, s.groups, s.act)
            secs += time.perf_counter() - t0
            fl += 2.0 * macs(s) * count / total
            npts += count
        return fl, secs, npts

    # calibrate: grow the sample until it takes at least half the budget
    # (a tiny first sample is dominated by fixed costs and overestimates the
    # time per point)
    frac = 2e-5
    fl, secs, npts = run(frac)
    for _ in range(4):
        if secs >= 0.5 * budget_s or frac >= 1.0:
            break
        frac = min(1.0, frac * min(100.0, budget_s / max(secs, 1e-3)))
        fl, secs, npts = run(frac)
    return fl, secs, npts, oracle.max_threads(0)


def cpu_baseline(layers, budget_s=12.0):
    fl, secs, npts, thr = oracle_sample(layers, budget_s)
    return {"value": round(fl / secs / 1e12, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"{npts} random output points across the {len(layers)} layers "
                      f"({fl / 1e9:.2f} GFLOP, {secs:.1f} s, fp64 nested loops, OpenMP)"}


def run_reference(args):
    from conv_workloads import generate
    layers = generate(args.workload)
    per_step_budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(layers, per_step_budget / 4, seed=1)
    fl_tot, s_tot, pts_tot, thr = 0.0, 0.0, 0, 1
    for k in range(args.steps):
        fl, secs, npts, thr = oracle_sample(layers, per_step_budget, seed=100 + k)
        fl_tot += fl
        s_tot += secs
        pts_tot += npts
    value = fl_tot / s_tot / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s_tot / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "layers": len(layers), "batch_per_gpu": layers[0].spec.n,
                   "note": "CPU oracle on a bounded random sample of output points per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{pts_tot} output points over {args.steps} steps "
                                   f"({fl_tot / 1e9:.2f} GFLOP in {s_tot:.1f} s)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true", help="skip timing the residual / concat / SPP rows")
    ap.add_argument("--no-layer-sets", action="store_true", help="skip timing the other layer sets")
    ap.add_argument("--only", default="",
                    help="run only these layers of the set (comma-separated names; for profiler captures)")
    ap.add_argument("--profile-pass", action="store_true",
                    help="run the layers eagerly (warmup + 1 passes, in order) for a profiler and print their "
                         "plans; no timing")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build()
    out = run_ours(args, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline and not args.profile_pass:
        from conv_workloads import generate
        out["cpu_baseline"] = cpu_baseline(generate(args.workload))
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
