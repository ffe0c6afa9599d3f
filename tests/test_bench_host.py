"""bench.py's host-side logic on CPU: the one-GPU rule (under
torch.distributed.run with more than one rank, rank 0 prints an
"unavailable" line, no rank loads the library), the reference arm printing
only on rank 0, the median over fresh processes, the forwarding of settings
to those processes, and the clock record's summary."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _bench(env_extra, *args, timeout=300):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          env=env, capture_output=True, text=True, timeout=timeout)


def test_more_than_one_rank_is_unavailable_on_rank_0():
    """No GPU here: had it touched CUDA or the library, the run would fail."""
    r = _bench({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}, "--gpus", "2",
               "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and "multicast" in d["unavailable"]
    assert "value" not in d


def test_more_than_one_rank_is_silent_elsewhere():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--gpus", "2")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_bench_loads_no_distributed_backend():
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert "init_process_group" not in src and "all_reduce" not in src


def test_reference_arm_is_silent_on_other_ranks():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference",
               "--steps", "1", "--warmup", "0", "--workload", "gemm_512")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_line_on_rank_0():
    r = _bench({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, "--impl", "reference",
               "--steps", "2", "--warmup", "1", "--workload", "gemm_512")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_median_leg_is_the_middle_value():
    import bench
    legs = [{"value": v, "i": i} for i, v in enumerate([3.0, 1.0, 2.0])]
    assert bench.median_leg(legs)["i"] == 2
    legs = [{"value": v, "i": i} for i, v in enumerate([4.0, 1.0, 3.0, 2.0])]
    assert bench.median_leg(legs)["value"] == 2.0          # lower middle
    assert bench.median_leg([{"value": 5.0}])["value"] == 5.0


def test_child_gets_the_parents_settings():
    import bench
    args = bench.parse(["--steps", "7", "--warmup", "4", "--workload", "gemm_ragged_3000x5000x4104",
                        "--acc", "f16", "--variant", "tc_pair_256x256_s6", "--tile-order", "static",
                        "--schedule", "whole", "--pdl", "off", "--cooldown", "1.5", "--graph"])
    argv = bench.child_argv(args)
    assert argv[1].endswith("bench.py") and argv[2] == "--child"
    child = bench.parse(argv[2:])
    assert child.child and child.graph
    for name in ("steps", "warmup", "workload", "acc", "variant", "tile_order", "schedule",
                 "pdl", "cooldown"):
        assert getattr(child, name) == getattr(args, name), name
    # a child never spawns children of its own, nor runs the e2e/sustained legs
    assert "--repeat" not in argv


def test_clock_summary_names_every_reason():
    """The clock record lists every clock-event reason seen (GPU idle aside),
    unnamed bits by value, with the minimum and 10th-percentile SM clock."""
    import torch
    import bench
    s = bench.ClockSampler(torch.device("cpu"))
    s.samples = ([(2070.0, 300.0, 0x0)] * 16 + [(1320.0, 360.0, 0x4 | 0x10)] * 3 +
                 [(2070.0, 100.0, 0x1 | 0x400)])
    d = s.summary()
    assert d["reasons"] == ["0x400", "sw_power_cap", "sync_boost"]
    assert d["sm_mhz"] == 2070.0 and d["sm_min_mhz"] == 1320.0
    assert d["sm_p10_mhz"] == 1320.0
    assert d["samples"] == 20 and d["power_w_max"] == 360.0
    s.samples = [(2070.0, 300.0, 0x1)] * 5
    assert s.summary()["reasons"] == []


def test_kernel_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    """A recorded ncu traffic figure is keyed by a hash of the kernel sources'
    code: comments and whitespace leave it unchanged, a code change moves it,
    and the committed records carry the current sources' hash."""
    import json
    import shutil
    import bench
    csrc = tmp_path / "dense_fp16_gemm_04_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "dense_fp16_gemm_04_gb300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("*.o", "*.so"))
    h0 = bench.kernel_source_hash()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash() == h0
    ptx = csrc / "ptx.cuh"
    text = ptx.read_text()
    ptx.write_text("// a comment\n" + text.replace("\n", "\n  \n", 3) + "\n/* block\n comment */\n")
    assert bench.kernel_source_hash() == h0
    ptx.write_text(text + "\nstatic const int kProbe = 1;\n")
    assert bench.kernel_source_hash() != h0
    monkeypatch.undo()
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        records = json.load(f)
    assert records and all(r["source_hash"] == h0 for r in records.values())
