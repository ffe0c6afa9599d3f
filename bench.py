#!/usr/bin/env python3
"""Benchmark of the GB300 dense fp16 GEMM, C = A @ B.T (K-major operands).

One step = one C = A @ B.T over the whole workload (default: M = N = K = 8192,
fp32 accumulation, fp16 output), inputs resident in HBM.  Prints ONE JSON line
with TFLOP/s = 2*M*N*K / t, the roofline of the GEMM kernel against the
measured dense tensor peak, the SM clock the kernel itself ran at (its own
clock record) and the cycles it took per k-block, a seconds-long sustained
run against the sustained peak, an end-to-end number through the host-buffer
entry point (host<->device copies inside the timed region), and the CPU
oracle timed on a bounded sample of the same workload.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--acc f32|f16] [--repeat R]

Protocol of the headline number (tilus "Four Consumers, FP16 Accumulation,
and a TMA Epilogue", section "Performance"): R (default 3) fresh processes,
each waiting a cool-down (default 3 s) and then timing K back-to-back steps
with CUDA events; `value` is the median of the R.

--impl reference times the CPU oracle (the plain fp64 triple loop), on the
host cores, on bounded row samples of the same workload.  The library is for
one GPU: its ragged-K kernel multicasts TMA loads inside a cluster, which is
kept out of any multi-GPU run, so under torch.distributed.run with N > 1 rank
0 prints an "unavailable" line and no rank loads the library.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

import gemm_workloads as wl

METRIC = "fp16 GEMM TFLOP/s (2MNK/t) and % of GB300 dense fp16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_TFLOPS = 1900.0   # used only when the measured-peaks file is absent
DENSE_FLOP_PER_CLK_SM = 8192   # fp16 tcgen05 rate per SM per clock (measured, see roofline note)
MULTI_GPU_UNAVAILABLE = (
    "single-GPU library: its ragged-K kernel (tc_pair_mc_256x256_s6) multicasts TMA loads "
    "within a cluster, which is kept out of multi-GPU runs; the GEMM has no exchange step")

# Arguments a measuring child process inherits from its parent.
_CHILD_ARGS = ("steps", "warmup", "workload", "shape", "layout", "acc", "variant", "tile_order",
               "schedule", "pdl", "cooldown")


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gemm_8192", choices=list(wl.WORKLOADS))
    p.add_argument("--shape", default=None,
                   help="MxNxK: time this shape instead (seeded N(0,1)*K^-1/4 inputs, seed 0)")
    p.add_argument("--layout", default="kk", choices=["kk", "kn", "mk", "mn"],
                   help="storage of A and B: k = K-contiguous, m/n = M/N-contiguous")
    p.add_argument("--acc", default="f32", choices=["f32", "f16"])
    p.add_argument("--variant", default=None, help="force a kernel variant by name")
    p.add_argument("--tile-order", default="auto", choices=["auto", "static", "dynamic"],
                   help="order of whole tiles over the persistent units (results do not depend on it)")
    p.add_argument("--schedule", default="auto", choices=["auto", "whole", "streamk"],
                   help="work schedule: automatic, whole tiles only, or a stream-K share whenever possible")
    p.add_argument("--pdl", default="on", choices=["on", "off"],
                   help="programmatic dependent launch of consecutive GEMMs")
    p.add_argument("--graph", action="store_true",
                   help="capture the K timed launches in one CUDA graph (GPU time without "
                        "per-call host overhead; for small shapes)")
    p.add_argument("--repeat", type=int, default=3,
                   help="fresh processes timing the K steps; the headline value is their median")
    p.add_argument("--cooldown", type=float, default=3.0,
                   help="seconds of idle GPU before each process's timed steps")
    p.add_argument("--sustained-s", type=float, default=4.0,
                   help="seconds of back-to-back steps for the sustained leg (0 = skip)")
    p.add_argument("--child", action="store_true",
                   help="internal: time the K steps once and print that leg as JSON")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=0,
                   help="oracle sample size in rows (0 = sized for ~10 s)")
    return p.parse_args(argv)


def child_argv(args):
    """Command line of a child process that times the K steps once."""
    argv = [sys.executable, os.path.abspath(__file__), "--child"]
    for name in _CHILD_ARGS:
        v = getattr(args, name)
        if v is None:
            continue
        argv += ["--" + name.replace("_", "-"), str(v)]
    if args.graph:
        argv.append("--graph")
    return argv


def median_leg(legs):
    """The leg whose value is the median of the legs' values (the lower
    middle one for an even count)."""
    ranked = sorted(legs, key=lambda d: d["value"])
    return ranked[(len(ranked) - 1) // 2]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        # fp16 and bf16 dense tensor rates are nominally equal (1:1)
        return {"tflops": float(d["bf16_tflops"]), "tflops_sustained":
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"tflops": FALLBACK_TFLOPS, "tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, polled through NVML
    (read-only queries) on a background thread while the timed region runs.
    If NVML cannot be loaded the clocks are reported as unavailable."""

    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*); any other
    # bit except GPU idle (0x1) is reported by its value.
    REASONS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    IDLE = 0x1

    def __init__(self, torch_device, period_s: float = 0.002):
        self.period = period_s
        self.samples = []          # (sm_mhz, power_w, reasons_mask)
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            self._open_nvml(torch_device)
        except Exception:
            self._nvml = None

    def _open_nvml(self, dev):
        import ctypes
        import threading
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(dev).uuid)
            ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev.index or 0),
                                                       ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint(0)
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._handle, self._ct, self._threading = nv, h, ctypes, threading

    def _poll(self):
        ct, nv, h = self._ct, self._nvml, self._handle
        mhz, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            a = nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz))
            b = nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
            c = nv.nvmlDeviceGetCurrentClocksEventReasons(h, ct.byref(rs))
            if a == 0:
                self.samples.append((float(mhz.value), mw.value / 1000.0 if b == 0 else None,
                                     rs.value if c == 0 else 0))
            self._stop.wait(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._stop = self._threading.Event()
            self._thread = self._threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml" if self._nvml else "unavailable"}
        sm = [x[0] for x in self.samples]
        reasons = set()
        for _, _, mask in self.samples:
            for bit, name in self.REASONS.items():
                if mask & bit:
                    reasons.add(name)
            other = mask & ~(self.IDLE | sum(self.REASONS))
            if other:
                reasons.add("0x%x" % other)
        power = [x[1] for x in self.samples if x[1] is not None]
        ranked = sorted(sm)
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": ranked[0],
                "sm_p10_mhz": ranked[len(ranked) // 10],
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "source": "nvml, polled every %.0f ms in the timed region" % (self.period * 1e3)}


def cpu_oracle_rate(w, rows_req=0, steps=1, a=None, b=None):
    """Time the CPU oracle on `rows` seeded rows of the workload; returns
    (TFLOP/s, threads used, sample description, seconds per step list)."""
    import oracle
    if a is None:
        a, b = wl.inputs_for(w)
    if rows_req <= 0:
        # size the sample for about 10 s on this host: probe 8 rows first
        probe = wl.sample_indices(w.M, 8, 99)
        t0 = time.perf_counter()
        oracle.gemm_rows_f64(a, b, probe)
        per_row = (time.perf_counter() - t0) / len(probe)
        rows_req = int(max(16, min(w.M, 10.0 / max(per_row, 1e-9))))
    rows = wl.sample_indices(w.M, rows_req, 4242)
    times, used = [], 0
    for _ in range(steps):
        t0 = time.perf_counter()
        _, used = oracle.gemm_rows_f64(a, b, rows, return_threads=True)
        times.append(time.perf_counter() - t0)
    flops = 2.0 * len(rows) * w.N * w.K
    rate = flops / statistics.median(times) / 1e12
    sample = (f"{len(rows)} seeded rows of C ({len(rows)}x{w.N}, K={w.K}) of {w.name}, "
              f"fp64 triple loop")
    return rate, used, sample, times


def resolve_workload(args):
    """The named workload, or an ad-hoc one from --shape."""
    if args.shape:
        M, N, K = (int(v) for v in args.shape.lower().split("x"))
        return wl.Workload(f"shape_{M}x{N}x{K}", M, N, K, 0, "normal", ("f32", "f16"))
    return wl.WORKLOADS[args.workload]


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = resolve_workload(args)
    a, b = wl.inputs_for(w)
    # each step: a bounded row sample sized so warmup+steps end in a few minutes
    budget_s = 150.0
    nsteps = args.steps + args.warmup
    probe = wl.sample_indices(w.M, 8, 99)
    import oracle
    t0 = time.perf_counter()
    oracle.gemm_rows_f64(a, b, probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    rows = int(max(8, min(w.M, budget_s / max(nsteps, 1) / max(per_row, 1e-9))))
    if args.cpu_rows > 0:
        rows = args.cpu_rows
    if args.warmup:
        cpu_oracle_rate(w, rows, steps=args.warmup, a=a, b=b)
    rate, used, sample, times = cpu_oracle_rate(w, rows, steps=args.steps, a=a, b=b)
    ms = statistics.median(times) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "acc": args.acc,
                   "sample": sample},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class Setup:
    """The library, a plan with the requested settings, the workload's
    operands on the GPU and the step function every timed leg runs."""

    def __init__(self, args):
        import torch

        import dense_fp16_gemm_04_gb300 as g

        self.torch, self.g = torch, g
        torch.cuda.set_device(0)
        self.dev = dev = torch.device("cuda", 0)
        g.build()
        self.plan = plan = g.Plan(0)
        if args.variant:
            plan.set_variant(args.variant)
        plan.set_tile_order(args.tile_order)
        plan.set_schedule(args.schedule)
        plan.set_pdl(args.pdl == "on")
        plan.set_clock_record(True)
        self.w = w = resolve_workload(args)
        self.acc = args.acc
        self.a_np, self.b_np = wl.inputs_for(w)
        la = g.MN_CONTIGUOUS if args.layout[0] == "m" else g.K_CONTIGUOUS
        lb = g.MN_CONTIGUOUS if args.layout[1] == "n" else g.K_CONTIGUOUS
        self.kk = la == g.K_CONTIGUOUS and lb == g.K_CONTIGUOUS
        self.la, self.lb = la, lb
        a = torch.from_numpy(self.a_np if la == g.K_CONTIGUOUS
                             else np.ascontiguousarray(self.a_np.T)).to(dev)
        b = torch.from_numpy(self.b_np if lb == g.K_CONTIGUOUS
                             else np.ascontiguousarray(self.b_np.T)).to(dev)
        c = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # Operands come from HBM in every step.  When A and B together are
        # larger than L2 one set streams through it; otherwise the steps
        # rotate over copies of A, B and C, enough that more than twice L2 is
        # touched between two uses of the same copy.
        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
        ab_bytes = (a.numel() + b.numel()) * 2
        set_bytes = ab_bytes + c.numel() * 2
        self.n_sets = n_sets = (1 if ab_bytes > l2_bytes else
                                min(4096, -(-2 * l2_bytes // max(set_bytes, 1)) + 1))
        sets = [(a, b, c)] + [(a.clone(), b.clone(), torch.empty_like(c))
                              for _ in range(n_sets - 1)]
        self.sets = sets
        self.ptrs = [(x.data_ptr(), y.data_ptr(), z.data_ptr()) for x, y, z in sets]
        self.l2_note = (
            "inputs larger than L2 (A+B = %d MB vs %d MB L2), no flush"
            % (ab_bytes >> 20, l2_bytes >> 20) if n_sets == 1 else
            "%d rotating copies of A, B and C (%d MB in all vs %d MB L2): operands from HBM "
            "every step, no flush" % (n_sets, (n_sets * set_bytes) >> 20, l2_bytes >> 20))

    def step(self, i, stream_handle=None):
        sh = self.stream.cuda_stream if stream_handle is None else stream_handle
        aptr, bptr, cptr = self.ptrs[i % self.n_sets]
        w = self.w
        if self.kk:
            self.plan.run_ptr(aptr, bptr, cptr, w.M, w.N, w.K, self.acc, sh)
        else:
            self.plan.run_ex_ptr(aptr, self.la, bptr, self.lb, cptr, w.M, w.N, w.K, self.acc, sh)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    def kblocks_per_unit(self):
        """k-blocks (64 deep) each persistent unit runs per launch, and the
        cycles one k-block of that unit's tile needs at the dense rate."""
        w = self.w
        d = self.plan.describe(w.M, w.N, w.K, self.acc)
        num_kb = -(-w.K // 64)
        total = d["dp_tiles"] * num_kb + d["sk_iters"]
        units = max(1, d["units"])
        vi = self.g.variant_info(d["variant"])
        ideal = vi["tile_m"] * vi["tile_n"] * 64 * 2 / (DENSE_FLOP_PER_CLK_SM * vi["ctas"])
        return total / units, ideal, d


def device_leg(args, su):
    """Warm up, wait the cool-down, then time K back-to-back steps with one
    CUDA event pair on the launching stream; NVML clocks are sampled during
    the steps and the kernels' own clock record is read after them."""
    torch, plan = su.torch, su.plan
    n_warm = max(args.warmup, 3)
    for i in range(n_warm):
        su.step(i)
    plan.check_error()
    graph = None
    if args.graph:
        cap = torch.cuda.Stream(su.dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                su.step(n_warm + i, cap.cuda_stream)
        graph.replay()
        su.sync()
    if args.cooldown > 0:
        time.sleep(args.cooldown)
    plan.kernel_clock()                      # start the clock record from zero
    launches0 = plan.launch_count
    sampler = ClockSampler(su.dev)
    su.sync()
    with sampler:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(su.stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                su.step(n_warm + i)
        e1.record(su.stream)
        su.sync()
    launches = plan.launch_count - launches0 if graph is None else args.steps
    plan.check_error()
    kclk = plan.kernel_clock()
    ms = e0.elapsed_time(e1) / args.steps
    w = su.w
    kb_unit, ideal, d = su.kblocks_per_unit()
    cyc = ms * 1e-3 * kclk["mhz"] * 1e6 if kclk["mhz"] else None
    return {"leg": "device", "value": w.flops / (ms * 1e-3) / 1e12, "ms_per_step": ms,
            "steps": args.steps, "gpu_launches": int(launches), "clocks": sampler.summary(),
            "kernel_clock": {"mhz": kclk["mhz"], "launches": kclk["launches"],
                             "source": "the kernel's own record: %clock64 over %globaltimer "
                                       "across CTA 0's lifetime, summed over the timed launches"},
            "cycles_per_kblock": cyc / kb_unit if cyc else None,
            "ideal_cycles_per_kblock": ideal, "kblocks_per_unit": kb_unit,
            "units": d["units"], "variant": d["variant"], "grid_ctas": d["grid_ctas"]}


def sustained_leg(args, su, seconds, step_ms):
    """Back-to-back steps for about `seconds` between one CUDA event pair,
    long enough for the board's power limit to set the SM clock."""
    torch, plan = su.torch, su.plan
    n = max(args.steps, int(seconds * 1e3 / max(step_ms, 1e-3)) + 1)
    for i in range(3):
        su.step(i)
    su.sync()
    plan.kernel_clock()
    sampler = ClockSampler(su.dev, period_s=0.02)
    with sampler:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(su.stream)
        for i in range(n):
            su.step(i)
        e1.record(su.stream)
        su.sync()
    plan.check_error()
    kclk = plan.kernel_clock()
    total_ms = e0.elapsed_time(e1)
    return {"value": n * su.w.flops / (total_ms * 1e-3) / 1e12, "unit": UNIT,
            "seconds": total_ms * 1e-3, "steps": n, "ms_per_step": total_ms / n,
            "clocks": sampler.summary(), "kernel_mhz": kclk["mhz"]}


def e2e_leg(args, su):
    """The same product through gemm_run_host: pinned host buffers, the
    host->device copies of A and B and the device->host copy of C inside
    every timed step (the call is synchronous)."""
    torch, plan, w = su.torch, su.plan, su.w
    ha = torch.from_numpy(su.a_np).pin_memory()
    hb = torch.from_numpy(su.b_np).pin_memory()
    hc = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    hp = (ha.data_ptr(), hb.data_ptr(), hc.data_ptr())
    sh = su.stream.cuda_stream
    for _ in range(2):
        plan.run_host_ptr(*hp, w.M, w.N, w.K, args.acc, sh)
    e_steps = max(3, min(args.steps, 10))
    su.sync()
    t0 = time.perf_counter()
    marks = []
    for _ in range(e_steps):
        plan.run_host_ptr(*hp, w.M, w.N, w.K, args.acc, sh)  # synchronous
        marks.append(time.perf_counter())
    dt = marks[-1] - t0
    step_ms = sorted((b - a) * 1e3 for a, b in zip([t0] + marks[:-1], marks))
    return {"value": e_steps * w.flops / dt / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": int(su.a_np.nbytes + su.b_np.nbytes),
            "d2h_bytes_per_step": int(w.M * w.N * 2),
            "ms_per_step": dt / e_steps * 1e3, "steps": e_steps,
            # the steps one by one: a host-link hiccup shows here
            "step_ms": {"min": step_ms[0], "median": step_ms[len(step_ms) // 2],
                        "max": step_ms[-1]}}


def run_child(args):
    su = Setup(args)
    leg = device_leg(args, su)
    su.plan.close()
    print(json.dumps(leg), flush=True)
    return 0


def run_ours(args):
    rank, world, _ = dist_env()
    if world > 1:
        # One GPU only (see the module docstring): nothing is loaded.
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "n_gpus": world,
                              "higher_is_better": True, "unavailable": MULTI_GPU_UNAVAILABLE}),
                  flush=True)
        return 0
    if args.child:
        return run_child(args)

    # ---------------------------------------- headline: R fresh processes --
    legs = []
    if args.repeat > 1:
        for _ in range(args.repeat):
            r = subprocess.run(child_argv(args), capture_output=True, text=True)
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise SystemExit(f"measuring process failed (rc {r.returncode})")
            legs.append(json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1]))
    su = Setup(args)
    if args.repeat <= 1:
        legs.append(device_leg(args, su))
    head = median_leg(legs)
    w = su.w

    peaks = measured_peaks()
    clocks = head["clocks"]
    # The burst peak for a kernel timed alone; once the power cap has acted
    # inside the timed region (a long step), the sustained one.
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    peak = peaks["tflops_sustained"] if capped else peaks["tflops"]
    peak_source = "%s bf16 %s (fp16 1:1)" % (peaks["source"],
                                            "sustained: power cap active" if capped else "burst")
    kernel_ms = head["ms_per_step"]
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    # Roofline of the kernel: algorithmic bytes 2(MK + NK + MN) against the
    # measured copy bandwidth when the arithmetic intensity is below the
    # ridge (C with few rows: HBM-bound), else FLOP against the tensor peak.
    alg_bytes = 2.0 * (w.M * w.K + w.N * w.K + w.M * w.N)
    hbm_bound = w.flops / alg_bytes < peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": alg_bytes / (kernel_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_source": peaks["source"] + " copy bandwidth"}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "peak_source": peak_source}
    roof["frac"] = roof["achieved"] / roof["peak"]

    # ------------------------------------------------ sustained, end to end --
    sustained = None
    if args.sustained_s > 0:
        sustained = sustained_leg(args, su, args.sustained_s, kernel_ms)
        if hbm_bound:
            # the same bound as the headline's roofline: bytes against the copy rate
            gbs = alg_bytes / (sustained["ms_per_step"] * 1e-3) / 1e9
            sustained.update({"bound": "hbm", "achieved": gbs, "achieved_unit": "GB/s",
                              "peak": peaks["hbm_gbs"],
                              "peak_source": peaks["source"] + " copy bandwidth",
                              "frac": gbs / peaks["hbm_gbs"]})
        else:
            sustained.update({"bound": "tensor", "peak": peaks["tflops_sustained"],
                              "peak_source": peaks["source"] + " bf16 sustained (fp16 1:1)",
                              "frac": sustained["value"] / peaks["tflops_sustained"]})
    e2e = e2e_leg(args, su) if not args.no_e2e and args.layout == "kk" else None

    cpu = None
    if not args.no_cpu_baseline:
        rate, used, sample, _ = cpu_oracle_rate(w, args.cpu_rows, steps=1, a=su.a_np, b=su.b_np)
        cpu = {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample}

    # The recorded ncu traffic is for the automatic settings only.
    defaults = (args.layout == "kk" and args.schedule == "auto" and args.tile_order == "auto"
                and args.pdl == "on" and not args.variant)
    traffic = _recorded_traffic(w.name, args.acc, head["variant"]) if defaults else None
    kclk = dict(head["kernel_clock"])
    kclk["cycles_per_kblock"] = head["cycles_per_kblock"]
    kclk["ideal_cycles_per_kblock"] = head["ideal_cycles_per_kblock"]
    kclk["kblocks_per_unit"] = head["kblocks_per_unit"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": kernel_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "M": w.M, "N": w.N, "K": w.K,
                   "acc": args.acc, "layout": args.layout, "variant": head["variant"],
                   "grid_ctas": head["grid_ctas"], "l2": su.l2_note, "parallelism": "single GPU",
                   "launch": "CUDA graph of the K steps" if args.graph else "one call per step",
                   "schedule": args.schedule, "tile_order": args.tile_order, "pdl": args.pdl},
        "repeats": {"n": len(legs), "values": [d["value"] for d in legs],
                    "kernel_mhz": [d["kernel_clock"]["mhz"] for d in legs],
                    "how": ("median of %d fresh processes, each after a %.0f s cool-down"
                            % (len(legs), args.cooldown)) if len(legs) > 1 else
                           "one process, after a %.0f s cool-down" % args.cooldown},
        "pct_of_peak": head["value"] / peak,
        "roofline": {**roof, "traffic": traffic},
        "clocks": clocks, "kernel_clock": kclk,
        "cycles_per_kblock": head["cycles_per_kblock"],
        "sustained": sustained, "e2e": e2e, "gpu_launches": head["gpu_launches"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    su.plan.close()
    return 0


def kernel_source_hash() -> str:
    """Hash of the CUDA sources' code (comments and whitespace removed): a
    recorded ncu traffic figure is used only while the code it was measured
    on is unchanged."""
    import glob
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_04_gb300", "csrc")
    for path in sorted(glob.glob(os.path.join(csrc, "*.cu*"))):
        with open(path, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(os.path.basename(path).encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _recorded_traffic(workload, acc, variant):
    """DRAM bytes (read + write) per launch from the committed ncu summary of
    this kernel variant and workload, or None if none was recorded for the
    current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{variant}/{workload}/{acc}")
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return int(e["dram_bytes_per_launch"])


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
