"""The dynamic order of whole tiles against the static round robin.

In the dynamic order each unit's first whole tile is fixed and its later
ones come from a global ticket counter (taken by the leader CTA's scheduler
warp and handed to every role of the cluster through a two-slot ring in
shared memory).  Which unit computes a tile never changes the tile's own
sequence of MMAs, and the stream-K share and its fix-up order do not depend
on the order of whole tiles, so the two orders must agree bit for bit.  The
counters must come back to zero after every launch (alternating shapes,
repeated launches) and after a launch that gave up."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import assert_close

pytestmark = pytest.mark.gpu


def _plan(variant=None, order="auto", schedule="auto"):
    p = g.Plan(0)
    if variant:
        p.set_variant(variant)
    p.set_tile_order(order)
    p.set_schedule(schedule)
    return p


def _run(p, ta, tb, M, N, acc="f32", reps=1):
    outs = []
    for _ in range(reps):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        p.run(ta, tb, c, acc=acc)
        outs.append(c)
    p.check_error()
    return outs


# (variant, M, N, K, acc, schedule): several waves of whole tiles for each
# kernel form, with and without a stream-K share.
CASES = [
    ("tc_pair_256x256_s6", 4096, 4096, 512, "f32", "whole"),
    ("tc_pair_256x256_s6", 4096, 4096, 1032, "f32", "auto"),     # share + dynamic whole tiles
    ("tc_pair_256x256_s6", 2056, 8192, 1024, "f16", "auto"),
    ("tc_pair_mc_256x256_s6", 3000, 5000, 1032, "f32", "auto"),   # two-pair clusters
    ("tc_pair_256x128_s8", 2048, 4104, 520, "f32", "whole"),
    ("tc_single_128x256_s4", 2048, 4096, 256, "f32", "whole"),
    ("tc_single_128x64_s8", 1100, 2048, 264, "f32", "auto"),
    ("tc_swap_16x128_s11", 16, 40000, 256, "f32", "whole"),
    ("tc_swap_64x128_s8", 60, 24000, 264, "f16", "whole"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0][3:]}-{c[1]}x{c[2]}x{c[3]}-{c[4]}-{c[5]}")
def test_dynamic_order_matches_static(case):
    variant, M, N, K, acc, schedule = case
    a, b = wl.draw(M, N, K, seed=M + N + K)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ps, pd = _plan(variant, "static", schedule), _plan(variant, "dynamic", schedule)
    ref = _run(ps, ta, tb, M, N, acc)[0]
    got = _run(pd, ta, tb, M, N, acc, reps=3)
    for i, c in enumerate(got):
        assert torch.equal(c, ref), f"launch {i}: dynamic order differs from static"
    rows = wl.sample_indices(M, 24, 5)
    assert_close(got[-1].cpu().numpy()[rows], oracle.gemm_rows_f64(a, b, rows), acc, str(case))
    ps.close()
    pd.close()


def test_counters_return_to_zero_between_shapes():
    """Alternate shapes with different numbers of whole tiles on one plan:
    a counter left behind by one launch would skip or repeat tiles in the
    next, which the NaN-filled outputs and the static reference expose."""
    p, ps = _plan(order="dynamic"), _plan(order="static")
    cases = []
    for shape in [(4096, 4096, 256), (1024, 8192, 520), (2048, 2048, 64), (300, 520, 328)]:
        a, b = wl.draw(*shape, seed=sum(shape) + 1)
        ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
        cases.append((shape, ta, tb, _run(ps, ta, tb, shape[0], shape[1])[0]))
    for rnd in range(5):
        for (M, N, K), ta, tb, ref in cases:
            c = _run(p, ta, tb, M, N)[0]
            assert torch.equal(c, ref), f"{(M, N, K)} round {rnd}"
    p.close()
    ps.close()


def test_back_to_back_launches_without_sync():
    """Twenty launches queued back to back (programmatic dependent launch:
    each kernel's set-up overlaps the previous one's end, and its scheduler
    takes tickets only once that kernel is complete)."""
    M, N, K = 4096, 4096, 256
    a, b = wl.draw(M, N, K, seed=77)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ps, pd = _plan(order="static"), _plan(order="dynamic")
    ref = _run(ps, ta, tb, M, N)[0]
    outs = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(20)]
    for c in outs:
        pd.run(ta, tb, c)
    pd.check_error()
    for i, c in enumerate(outs):
        assert torch.equal(c, ref), f"launch {i}"
    ps.close()
    pd.close()


def test_automatic_choice_uses_dynamic_order_for_many_waves():
    """The automatic order is dynamic from 24 waves of whole tiles on (here
    64 x 32 = 2048 pair tiles, 27 waves over 76 pairs); either way the result
    is the static one."""
    M, N, K = 16384, 8192, 64
    a, b = wl.draw(M, N, K, seed=78)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    pa, ps = _plan(order="auto"), _plan(order="static")
    assert torch.equal(_run(pa, ta, tb, M, N)[0], _run(ps, ta, tb, M, N)[0])
    pa.close()
    ps.close()


def test_timeout_in_dynamic_order_leaves_a_usable_plan():
    """A launch that gives up (an injected never-declared stage) may leave
    the ticket counters mid-count; gemm_plan_check_error reports the timeout
    and resets them, and the next launch is exact."""
    M, N, K = 4096, 4096, 512
    a, b = wl.draw(M, N, K, seed=79)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ps, pd = _plan(order="static"), _plan(order="dynamic")
    ref = _run(ps, ta, tb, M, N)[0]
    pd.set_watchdog(timeout_ns=50_000_000, skip_k_block=0)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    pd.run(ta, tb, c)
    assert pd.check_error_status() == 5
    pd.set_watchdog(0, -1)
    for _ in range(2):
        assert torch.equal(_run(pd, ta, tb, M, N)[0], ref)
    ps.close()
    pd.close()


def test_graph_replay_in_dynamic_order():
    """A captured launch in the dynamic order replays correctly: the ticket
    counters are back at zero at the end of every launch, graph or not."""
    M, N, K = 4096, 4096, 256
    a, b = wl.draw(M, N, K, seed=80)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ps, pd = _plan(order="static"), _plan(order="dynamic")
    ref = _run(ps, ta, tb, M, N)[0]
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pd.run(ta, tb, c)               # first call outside the capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pd.run(ta, tb, c)
    for _ in range(4):
        c.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(c, ref)
    pd.check_error()
    ps.close()
    pd.close()


def test_set_tile_order_rejects_other_values(plan):
    with pytest.raises(g.GemmError):
        plan.set_tile_order(3)
