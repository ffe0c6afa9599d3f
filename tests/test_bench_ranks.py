"""The multi-rank side of bench.py on CPU: two gloo ranks, each with its own
time, must agree on the slowest rank's time, and the whole-job throughput is
ranks x steps x FLOP / that time.  Also: the reference arm prints only on
rank 0."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(1.5 if rank == 0 else 2.5, world)
    out[rank] = (t, bench.aggregate_tflops(world, 10, 1e12, t))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    t, tflops = out[0]
    assert t == 2.5
    assert tflops == pytest.approx(2 * 10 * 1e12 / 2.5 / 1e12)


def test_single_rank_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    assert bench.aggregate_tflops(1, 4, 2e12, 2.0) == pytest.approx(4.0)


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "gemm_512"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_line_on_rank_0():
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "gemm_512"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_shard_rows_cover_every_row_once():
    import dense_fp16_gemm_04_gb300 as g
    for M in [1, 7, 255, 256, 257, 3000, 8192, 16384, 100000]:
        for world in [1, 2, 3, 4, 8]:
            covered = []
            for rank in range(world):
                row0, rows = g.shard_rows(M, world, rank)
                assert rows >= 0 and (row0 % 256 == 0 or rows == 0 or row0 == M)
                covered.extend(range(row0, row0 + rows))
            assert covered == list(range(M)), (M, world)
    with pytest.raises(ValueError):
        g.shard_rows(10, 2, 2)


def _shard_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import dense_fp16_gemm_04_gb300 as g
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    row0, rows = g.shard_rows(3000, world, rank)
    mine = torch.zeros(3000, dtype=torch.int64)
    mine[row0:row0 + rows] = 1
    dist.all_reduce(mine)                      # every row owned exactly once
    out[rank] = bool((mine == 1).all())
    dist.destroy_process_group()


def test_two_gloo_ranks_split_rows_disjointly():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] and out[1]


def test_clock_summary_names_every_reason():
    """The clock record lists every clock-event reason seen (GPU idle aside),
    unnamed bits by value, with the minimum and 10th-percentile SM clock."""
    import torch
    sys.path.insert(0, ROOT)
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
