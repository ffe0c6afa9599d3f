"""Programmatic dependent launch: a GEMM launched right behind another one in
the same stream may start its set-up early, but it must not read or write
global memory before the previous kernel has completed.  Chains of dependent
GEMMs (read-after-write and write-after-read through the same buffers) are run
back to back with the overlap on and no synchronisation, and compared bit for
bit with the same chain run with plain stream ordering and a synchronisation
after every launch.  The kernel is deterministic, so any early read or write
shows up as a difference."""
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl

pytestmark = pytest.mark.gpu

# (M, K, schedule): square chains A[M,K] -> C[M,K] need N == K.
CHAINS = [
    (2048, 2048, "auto"),     # 256x256 pair tiles
    (384, 512, "auto"),       # 128x64 tiles (small problem)
    (16, 1024, "auto"),       # swapped roles (M <= 16)
    (1536, 1024, "streamk"),  # stream-K share on every launch: workspace reuse
]


def _chain(plan, a, bs, acc, sync):
    """x <- a; for each b: y = x . b^T, then x <- y written over the buffer the
    step before last read (write-after-read), so each launch depends on the
    previous one both ways."""
    x = a.clone()
    y = torch.empty_like(a)
    for b in bs:
        plan.run(x, b, y, acc=acc)
        if sync:
            torch.cuda.synchronize()
        x, y = y, x
    torch.cuda.synchronize()
    return x


@pytest.mark.parametrize("M,K,sched", CHAINS)
@pytest.mark.parametrize("acc", ["f32", "f16"])
def test_dependent_chain_matches_serialised_chain(M, K, sched, acc):
    if acc == "f16" and sched == "streamk":
        pytest.skip("fp16 accumulation never uses the stream-K share")
    a_np, _ = wl.draw(M, K, K, seed=71)
    bs = [torch.from_numpy(wl.draw(K, K, K, seed=72 + i)[1] * 0.5).cuda() for i in range(6)]
    a = torch.from_numpy(a_np).cuda()

    ref_plan = g.Plan(0)
    ref_plan.set_pdl(False)
    ref_plan.set_schedule(sched)
    ref = _chain(ref_plan, a, bs, acc, sync=True)
    ref_plan.check_error()

    plan = g.Plan(0)
    plan.set_schedule(sched)  # overlap on by default
    for _ in range(3):
        got = _chain(plan, a, bs, acc, sync=False)
        plan.check_error()
        assert torch.equal(got, ref), f"chain M={M} K={K} {sched} {acc} differs"
    assert not bool(torch.isnan(ref).any())


def test_mixed_variants_back_to_back():
    """Launches of different variants (and so different grids) follow each
    other without synchronisation: small, tall, skinny, then small again."""
    shapes = [(300, 520, 328), (2048, 2048, 1024), (16, 4096, 2048), (1000, 1000, 1000)]
    data = []
    for i, (M, N, K) in enumerate(shapes):
        a, b = wl.draw(M, N, K, seed=80 + i)
        data.append((torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()))

    ref_plan = g.Plan(0)
    ref_plan.set_pdl(False)
    refs = []
    for (a, b), (M, N, K) in zip(data, shapes):
        c = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ref_plan.run(a, b, c)
        torch.cuda.synchronize()
        refs.append(c)

    plan = g.Plan(0)
    outs = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            for (M, N, K) in shapes]
    for _ in range(2):
        for (a, b), c in zip(data, outs):
            plan.run(a, b, c)
    torch.cuda.synchronize()
    plan.check_error()
    for c, r, s in zip(outs, refs, shapes):
        assert torch.equal(c, r), f"shape {s}"


def test_set_pdl_rejects_other_values():
    plan = g.Plan(0)
    assert plan._lib.gemm_plan_set_pdl(plan._h, 2) == 1  # GEMM_ERR_INVALID_ARG
    assert plan._lib.gemm_plan_set_pdl(plan._h, -1) == 1
    plan.set_pdl(False)
    plan.set_pdl(True)
