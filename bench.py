#!/usr/bin/env python3
"""Benchmark of the GB300 dense fp16 GEMM, C = A @ B.T (K-major operands).

One step = one C = A @ B.T over the whole workload (default: M = N = K = 8192,
fp32 accumulation, fp16 output), inputs resident in HBM.  Prints ONE JSON line
with TFLOP/s = 2*M*N*K / t, the roofline of the GEMM kernel against the
measured dense tensor peak, an end-to-end number through the host-buffer
entry point (host<->device copies inside the timed region), and the CPU
oracle timed on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--acc f32|f16]

--impl reference times the CPU oracle (the plain fp64 triple loop), on the
host cores, on bounded row samples of the same workload.  For N > 1 (launched
under torch.distributed.run) every rank runs an independent replica of the
workload on its own GPU: the GEMM has no exchange step, so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
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


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gemm_8192", choices=list(wl.WORKLOADS))
    p.add_argument("--shape", default=None,
                   help="MxNxK: time this shape instead (seeded N(0,1)*K^-1/4 inputs, seed 0)")
    p.add_argument("--split", default="replicas", choices=["replicas", "m"],
                   help="N > 1: every rank runs the whole workload (replicas, weak scaling) or "
                        "its share of C's rows (m, strong scaling)")
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
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=0,
                   help="oracle sample size in rows (0 = sized for ~10 s)")
    return p.parse_args()


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


def run_ours(args):
    import torch
    import torch.distributed as dist

    import dense_fp16_gemm_04_gb300 as g

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    g.build()
    plan = g.Plan(local)
    if args.variant:
        plan.set_variant(args.variant)
    plan.set_tile_order(args.tile_order)
    plan.set_schedule(args.schedule)
    plan.set_pdl(args.pdl == "on")
    w_full = resolve_workload(args)
    w = w_full
    a_np, b_np = wl.inputs_for(w_full)
    if world > 1 and args.split == "m":
        # This rank's rows of A and C; B whole.  No exchange inside the product.
        row0, rows = g.shard_rows(w_full.M, world, rank)
        a_np = np.ascontiguousarray(a_np[row0:row0 + rows])
        w = wl.Workload(f"{w_full.name}_rows{row0}+{rows}", rows, w_full.N, w_full.K, w_full.seed,
                        w_full.dist, w_full.accs)
    la = g.MN_CONTIGUOUS if args.layout[0] == "m" else g.K_CONTIGUOUS
    lb = g.MN_CONTIGUOUS if args.layout[1] == "n" else g.K_CONTIGUOUS
    a = torch.from_numpy(a_np if la == g.K_CONTIGUOUS else np.ascontiguousarray(a_np.T)).to(dev)
    b = torch.from_numpy(b_np if lb == g.K_CONTIGUOUS else np.ascontiguousarray(b_np.T)).to(dev)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # Operands come from HBM in every step.  When A and B together are larger
    # than L2 one set streams through it; otherwise the steps rotate over
    # copies of A, B and C, enough that more than twice L2 is touched between
    # two uses of the same copy.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    ab_bytes = (a.numel() + b.numel()) * 2
    set_bytes = ab_bytes + c.numel() * 2
    n_sets = 1 if ab_bytes > l2_bytes else min(4096, -(-2 * l2_bytes // max(set_bytes, 1)) + 1)
    sets = [(a, b, c)] + [(a.clone(), b.clone(), torch.empty_like(c)) for _ in range(n_sets - 1)]
    ptrs = [(x.data_ptr(), y.data_ptr(), z.data_ptr()) for x, y, z in sets]
    l2_note = ("inputs larger than L2 (A+B = %d MB vs %d MB L2), no flush"
               % (ab_bytes >> 20, l2_bytes >> 20) if n_sets == 1 else
               "%d rotating copies of A, B and C (%d MB in all vs %d MB L2): operands from HBM "
               "every step, no flush" % (n_sets, (n_sets * set_bytes) >> 20, l2_bytes >> 20))

    def step(i, stream_handle=sh):
        aptr, bptr, cptr = ptrs[i % n_sets]
        if la == g.K_CONTIGUOUS and lb == g.K_CONTIGUOUS:
            plan.run_ptr(aptr, bptr, cptr, w.M, w.N, w.K, args.acc, stream_handle)
        else:
            plan.run_ex_ptr(aptr, la, bptr, lb, cptr, w.M, w.N, w.K, args.acc, stream_handle)

    n_warm = max(args.warmup, 3)
    for i in range(n_warm):
        step(i)
    plan.check_error()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ----------------------------------------------------- device-timed run --
    # One event pair around the K steps: no event sits between two launches,
    # so each GEMM's set-up may overlap the end of the previous one
    # (programmatic dependent launch, as in any back-to-back use).
    launches0 = plan.launch_count
    graph = None
    if args.graph:
        cap = torch.cuda.Stream(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                step(n_warm + i, cap.cuda_stream)
        graph.replay()
        torch.cuda.synchronize(dev)
        launches0 = plan.launch_count
    sampler = ClockSampler(dev)
    barrier()
    with sampler:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                step(n_warm + i)
        t_all1.record(stream)
        barrier()
    launches = plan.launch_count - launches0 if graph is None else args.steps
    plan.check_error()
    total_ms = reduce_max(t_all0.elapsed_time(t_all1), world, dev)
    per_launch_ms = [t_all0.elapsed_time(t_all1) / args.steps]
    clocks = sampler.summary()

    flops = float(w.flops)
    strong = world > 1 and args.split == "m"
    # replicas: every rank did its own full problem; m: the ranks together did one.
    value = (aggregate_tflops(1, args.steps, float(w_full.flops), total_ms * 1e-3) if strong
             else aggregate_tflops(world, args.steps, flops, total_ms * 1e-3))
    ms_per_step = total_ms / args.steps
    peaks = measured_peaks()
    # The burst peak for a kernel timed alone; once the power cap has acted
    # inside the timed region (a long step), the sustained one.
    sustained = "sw_power_cap" in (clocks.get("reasons") or [])
    peak = peaks["tflops_sustained"] if sustained else peaks["tflops"]
    peak_source = "%s bf16 %s (fp16 1:1)" % (peaks["source"],
                                            "sustained: power cap active" if sustained else "burst")
    kernel_ms = statistics.mean(per_launch_ms)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    # Roofline of the kernel: algorithmic bytes 2(MK + NK + MN) against the
    # measured copy bandwidth when the arithmetic intensity is below the
    # ridge (C with few rows: HBM-bound), else FLOP against the tensor peak.
    alg_bytes = 2.0 * (w.M * w.K + w.N * w.K + w.M * w.N)
    hbm_bound = flops / alg_bytes < peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": alg_bytes / (kernel_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_source": peaks["source"] + " copy bandwidth"}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "peak_source": peak_source}
    roof["frac"] = roof["achieved"] / roof["peak"]

    # ------------------------------------------------- end to end, host API --
    e2e = None
    if not args.no_e2e and args.layout == "kk":
        ha = torch.from_numpy(a_np).pin_memory()
        hb = torch.from_numpy(b_np).pin_memory()
        hc = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
        hp = (ha.data_ptr(), hb.data_ptr(), hc.data_ptr())
        for _ in range(2):
            plan.run_host_ptr(*hp, w.M, w.N, w.K, args.acc, sh)
        e_steps = max(3, min(args.steps, 10))
        barrier()
        t0 = time.perf_counter()
        marks = []
        for _ in range(e_steps):
            plan.run_host_ptr(*hp, w.M, w.N, w.K, args.acc, sh)  # synchronous
            marks.append(time.perf_counter())
        dt = reduce_max(marks[-1] - t0, world, dev)
        step_ms = sorted((b - a) * 1e3 for a, b in zip([t0] + marks[:-1], marks))
        e2e = {"value": (aggregate_tflops(1, e_steps, float(w_full.flops), dt) if strong
                         else aggregate_tflops(world, e_steps, flops, dt)), "unit": UNIT,
               "h2d_bytes_per_step": int(a_np.nbytes + b_np.nbytes),
               "d2h_bytes_per_step": int(w.M * w.N * 2),
               "ms_per_step": dt / e_steps * 1e3, "steps": e_steps,
               # this rank's steps one by one: a host-link hiccup shows here
               "step_ms": {"min": step_ms[0], "median": step_ms[len(step_ms) // 2],
                           "max": step_ms[-1]}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, used, sample, _ = cpu_oracle_rate(w, args.cpu_rows, steps=1, a=a_np, b=b_np)
        cpu = {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample}

    # The recorded ncu traffic is for the automatic settings only.
    defaults = (args.layout == "kk" and args.schedule == "auto" and args.tile_order == "auto"
                and args.pdl == "on")
    traffic = (_recorded_traffic(w.name, args.acc, plan.pick_variant(w.M, w.N, w.K, args.acc)[0])
               if defaults else None)
    variant, grid = plan.pick_variant(w.M, w.N, w.K, args.acc)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "strong" if strong else "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{w_full.name}: {w_full.describe()}", "M": w_full.M, "N": w.N, "K": w.K,
                   "acc": args.acc, "layout": args.layout, "variant": variant, "grid_ctas": grid,
                   "l2": l2_note,
                   "parallelism": (f"M split x{world}" if strong else f"replicas x{world}")
                                  if world > 1 else "single GPU",
                   "launch": "CUDA graph of the K steps" if graph is not None else "one call per step",
                   "schedule": args.schedule, "tile_order": args.tile_order, "pdl": args.pdl},
        "pct_of_peak": value / world / peak,
        "roofline": {**roof, "traffic": traffic},
        "clocks": clocks, "e2e": e2e, "gpu_launches": int(launches),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()
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


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, steps: int, flops_per_step: float, seconds: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of `flops_per_step`
    in `seconds` (the slowest rank's time)."""
    return world * steps * flops_per_step / seconds / 1e12


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
