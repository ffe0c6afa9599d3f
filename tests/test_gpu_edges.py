"""GPU edge cases: empty shapes, K == 0, argument rejection before any write,
out-of-bounds canaries, repeated launches, streams, and the host-buffer entry
point."""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import assert_close, run_gpu

pytestmark = pytest.mark.gpu

OK, INVALID, ALIGN = 0, 1, 2


def test_empty_M_or_N_is_a_no_op(plan):
    c = torch.full((4, 8), 7.0, dtype=torch.float16, device="cuda")
    a = torch.ones((4, 16), dtype=torch.float16, device="cuda")
    before = plan.launch_count
    assert plan.status_run(a.data_ptr(), a.data_ptr(), c.data_ptr(), 0, 8, 16) == OK
    assert plan.status_run(a.data_ptr(), a.data_ptr(), c.data_ptr(), 4, 0, 16) == OK
    assert plan.status_run(0, 0, 0, 0, 0, 0) == OK
    torch.cuda.synchronize()
    assert plan.launch_count == before
    assert bool((c == 7.0).all())


def test_K_zero_gives_zeros(plan):
    c = torch.full((33, 40), float("nan"), dtype=torch.float16, device="cuda")
    assert plan.status_run(0, 0, c.data_ptr(), 33, 40, 0) == OK
    plan.check_error()
    assert bool((c == 0).all())


def test_rejected_arguments_write_nothing(plan):
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    b = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    c = torch.full((64, 64), 3.0, dtype=torch.float16, device="cuda")
    pa, pb, pc = a.data_ptr(), b.data_ptr(), c.data_ptr()
    assert plan.status_run(pa, pb, pc, 64, 64, 60) == ALIGN          # K % 8
    assert plan.status_run(pa, pb, pc, 64, 60, 64) == ALIGN          # N % 8
    assert plan.status_run(pa + 2, pb, pc, 64, 64, 64) == ALIGN      # misaligned A
    assert plan.status_run(pa, pb + 8, pc, 64, 64, 64) == ALIGN      # misaligned B
    assert plan.status_run(pa, pb, pc + 4, 64, 64, 64) == ALIGN      # misaligned C
    assert plan.status_run(0, pb, pc, 64, 64, 64) == INVALID         # null A
    assert plan.status_run(pa, pb, 0, 64, 64, 64) == INVALID         # null C
    assert plan.status_run(pa, pb, pc, -1, 64, 64) == INVALID
    assert plan.status_run(pa, pb, pc, 64, 64, 1 << 31) == INVALID
    assert plan.status_run(pa, pb, pc, 64, 64, 64, acc=2) == INVALID
    assert plan.status_run(pa, pb, pa, 64, 64, 64) == INVALID        # C aliases A
    torch.cuda.synchronize()
    assert bool((c == 3.0).all())


def test_memory_of_no_device_or_the_host_is_refused(plan):
    """A, B and C must be device memory of the plan's device: host memory,
    pinned or pageable, is refused before any launch."""
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    c = torch.full((64, 64), 3.0, dtype=torch.float16, device="cuda")
    pinned = torch.ones((64, 64), dtype=torch.float16).pin_memory()
    pageable = np.ones((64, 64), dtype=np.float16)
    before = plan.launch_count
    for ha in (pinned.data_ptr(), pageable.ctypes.data):
        assert plan.status_run(ha, a.data_ptr(), c.data_ptr(), 64, 64, 64) == INVALID
        assert plan.status_run(a.data_ptr(), ha, c.data_ptr(), 64, 64, 64) == INVALID
        assert plan.status_run(a.data_ptr(), a.data_ptr(), ha, 64, 64, 64) == INVALID
        assert plan.status_run(0, 0, ha, 64, 64, 0) == INVALID       # K == 0 writes C
        st = plan._lib.gemm_run_ex(plan._h, ha, 1, a.data_ptr(), 0, c.data_ptr(), 64, 64, 64,
                                   0, torch.cuda.current_stream().cuda_stream)
        assert st == INVALID
    torch.cuda.synchronize()
    assert plan.launch_count == before
    assert bool((c == 3.0).all())


def test_kernel_clock_record():
    """With the clock record on, each GEMM launch adds one to it, with CTA
    0's lifetime in SM cycles and ns: their ratio is an SM clock the part
    can run at, and reading the record clears it.  Off (the default), the
    kernels leave it alone."""
    p = g.Plan(0)
    M = N = K = 1024
    a, b = wl.draw(M, N, K, seed=33)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for _ in range(3):
        p.run(ta, tb, c)
    assert p.kernel_clock()["launches"] == 0
    p.set_clock_record(True)
    for _ in range(5):
        p.run(ta, tb, c)
    r = p.kernel_clock()
    assert r["launches"] == 5 and r["cycles"] > 0 and r["ns"] > 0
    assert 200.0 < r["mhz"] < 3000.0, r
    assert p.kernel_clock()["launches"] == 0
    p.set_clock_record(False)
    p.run(ta, tb, c)
    assert p.kernel_clock()["launches"] == 0
    assert p._lib.gemm_plan_set_clock_record(p._h, 2) == INVALID
    p.check_error()
    p.close()


def test_writes_stay_inside_C(plan):
    """C sits inside a larger buffer of sentinels; a ragged shape must leave
    every byte before and after it untouched."""
    M, N, K = 203, 264, 200
    a, b = wl.draw(M, N, K, seed=31)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 1234.0, dtype=torch.float16, device="cuda")
    c = buf[guard:guard + M * N].view(M, N)
    plan.run(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), c)
    plan.check_error()
    host = buf.cpu()
    assert bool((host[:guard] == 1234.0).all()) and bool((host[guard + M * N:] == 1234.0).all())
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", "guarded")


def test_repeated_launches_stay_clean(plan):
    """Many back-to-back launches into a NaN-filled C: no NaN may ever appear
    (the symptom of a barrier placed inside a live TMA destination, tilus
    "A Minimal Hopper Matmul", Epilogue note)."""
    M, N, K = 1024, 2048, 1024
    a, b = wl.draw(M, N, K, seed=32)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    first = None
    for i in range(40):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(ta, tb, c, acc="f32" if i % 2 == 0 else "f16")
        if i % 2 == 0:
            if first is None:
                first = c.clone()
            else:
                assert torch.equal(c, first), f"launch {i} differs from launch 0"
        assert not bool(torch.isnan(c).any()), f"NaN in launch {i}"
    plan.check_error()


def test_side_stream(plan):
    M, N, K = 384, 512, 256
    a, b = wl.draw(M, N, K, seed=33)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    s = torch.cuda.Stream()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    with torch.cuda.stream(s):
        plan.run(ta, tb, c)
    s.synchronize()
    plan.check_error()
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", "side stream")


@pytest.mark.parametrize("acc", ["f32", "f16"])
def test_host_entry_point_matches_device_entry_point(acc):
    """gemm_run_host pipelines row chunks; with whole-tile schedules every tile
    is computed exactly as by gemm_run, so the results agree bit for bit."""
    p = g.Plan(0)
    p.set_schedule("whole")
    M, N, K = 700, 1032, 520
    a, b = wl.draw(M, N, K, seed=34)
    dev = run_gpu(p, a, b, acc)
    ha = torch.from_numpy(a).pin_memory()
    hb = torch.from_numpy(b).pin_memory()
    hc = torch.empty((M, N), dtype=torch.float16).pin_memory()
    p.run_host(ha, hb, hc, acc=acc)
    assert np.array_equal(hc.numpy().view(np.uint16), dev.view(np.uint16))
    # pageable numpy buffers work too
    out = np.empty((M, N), np.float16)
    p.run_host(a, b, out, acc=acc)
    assert np.array_equal(out.view(np.uint16), dev.view(np.uint16))
    p.close()


def test_host_entry_point_ragged_many_chunks(plan):
    """A ragged shape split into several row chunks (and, per chunk, whatever
    schedule the plan picks) against the oracle on sampled rows."""
    w = wl.WORKLOADS["gemm_ragged_3000x5000x4104"]
    a, b = wl.inputs_for(w)
    hc = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    plan.run_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(), hc)
    rows = wl.sample_indices(w.M, 64, 71)
    got = hc.numpy()[rows].astype(np.float64)
    assert_close(got, oracle.gemm_rows_f64(a, b, rows), "f32", "run_host ragged")


def test_host_entry_point_many_row_chunks(plan):
    """M = 9000 is cut into nine row chunks (1024 rows each, the last one
    ragged), each multiplied as soon as it has arrived; every row of C must
    come back, checked on sampled rows and on the last rows."""
    M, N, K = 9000, 520, 1032
    a, b = wl.draw(M, N, K, seed=72)
    hc = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    plan.run_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(), hc)
    rows = np.unique(np.concatenate([wl.sample_indices(M, 64, 73), np.arange(M - 8, M)]))
    got = hc.numpy()[rows].astype(np.float64)
    assert_close(got, oracle.gemm_rows_f64(a, b, rows), "f32", "run_host nine chunks")
    assert np.isfinite(hc.numpy()).all()


def test_host_entry_point_two_dimensional_blocks(plan):
    """MN / (M + N) >= 6144 switches gemm_run_host to cutting both A and B
    into row chunks: here 6 x 6 blocks of C with ragged last blocks in both
    directions, each multiplied as its two chunks arrive and copied back
    with a strided copy.  Every element must come back: sampled rows and
    columns against the oracle, all finite."""
    M, N, K = 12500, 13000, 72
    a, b = wl.draw(M, N, K, seed=74)
    hc = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    plan.run_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(), hc)
    c = hc.numpy()
    assert np.isfinite(c).all()
    rows = np.unique(np.concatenate([wl.sample_indices(M, 48, 75), [0, 2303, 2304, M - 1]]))
    cols = np.unique(np.concatenate([wl.sample_indices(N, 48, 76), [0, 2303, 2304, N - 1]]))
    assert_close(c[rows].astype(np.float64), oracle.gemm_rows_f64(a, b, rows), "f32", "2-D rows")
    assert_close(c[:, cols].astype(np.float64), oracle.gemm_cols_f64(a, b, cols), "f32", "2-D cols")


def test_host_entry_point_empty_and_zero_K(plan):
    """gemm_run_host on the degenerate shapes: K = 0 returns the empty sum
    (zeros) through the copy-out path; M = 0 or N = 0 touches nothing; a
    misaligned N is refused before anything is written."""
    for acc in ("f32", "f16"):
        out = np.full((40, 24), np.nan, np.float16)
        plan.run_host(np.zeros((40, 0), np.float16), np.zeros((24, 0), np.float16), out, acc=acc)
        assert np.array_equal(out.view(np.uint16), np.zeros((40, 24), np.uint16))
    out = np.full((0, 24), np.nan, np.float16)
    plan.run_host(np.zeros((0, 16), np.float16), np.ones((24, 16), np.float16), out)
    keep = np.full((40, 0), np.nan, np.float16)
    plan.run_host(np.ones((40, 16), np.float16), np.zeros((0, 16), np.float16), keep)
    bad = np.full((8, 12), np.nan, np.float16)
    with pytest.raises(g.GemmError):
        plan.run_host(np.ones((8, 16), np.float16), np.ones((12, 16), np.float16), bad)
    assert np.isnan(bad).all()


def test_gemm_convenience_wrapper(plan):
    a, b = wl.draw(256, 264, 128, seed=35)
    c = g.gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", "gemm()")


def test_variant_choice_and_launch_count(plan):
    name, grid = plan.pick_variant(8192, 8192, 8192)
    assert name in g.variant_names() and grid >= 1
    n0 = plan.launch_count
    run_gpu(plan, *wl.draw(128, 128, 64, seed=36))
    assert plan.launch_count == n0 + 1


def test_cuda_graph_capture_and_replay():
    """gemm_run only enqueues one kernel on the caller's stream (the tensor
    maps travel as kernel parameters and the stream-K counters reset
    themselves), so a captured call replays correctly, stream-K share
    included."""
    M, N, K = 4096, 4096, 4096          # 256 pair tiles: whole tiles + a stream-K share
    a, b = wl.draw(M, N, K, seed=37)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    p = g.Plan(0)
    assert p.describe(M, N, K)["sk_units"] > 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p.run(ta, tb, c)                 # first call outside the capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        p.run(ta, tb, c)
    rows = wl.sample_indices(M, 48, 38)
    ref = oracle.gemm_rows_f64(a, b, rows)
    for _ in range(3):
        c.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close(c.cpu().numpy()[rows], ref, "f32", "graph replay")
    p.check_error()
    p.close()
