"""The two-pair cluster kernel (tc_pair_mc_256x256_s6): two CTA pairs compute
neighbouring 256 x 256 tiles of one tile-row, and each CTA loads half of its
pair's A rows and multicasts it into the same position of both pairs.

Each pair issues exactly the MMAs of the one-pair kernel, in the same order,
on the same data, so with whole tiles (no stream-K share) the two kernels
must agree bit for bit.  Any stage consumed before the other pair's half of
A has landed shows up as a difference; the same launch is repeated many
times to give such a race every chance.  The general parity, stream-K,
layout, edge and watchdog tests cover this variant through the shared
variant list."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import assert_close

pytestmark = pytest.mark.gpu

MC = "tc_pair_mc_256x256_s6"
PAIR = "tc_pair_256x256_s6"

# (M, N, K): the ragged workload; an odd number of 256-column tiles (the
# second pair of the last unit has no columns of C); one k-block; a single
# unit tile; several tile-rows with a ragged K tail; fewer rows than one
# tile with a last k-block of 8 (one of its four 16-deep MMA steps used).
SHAPES = [(3000, 5000, 4104), (600, 1280, 520), (300, 760, 64), (256, 512, 1024),
          (1100, 2056, 2056), (200, 520, 1032)]


def _plan(variant, schedule):
    p = g.Plan(0)
    p.set_variant(variant)
    p.set_schedule(schedule)
    return p


@pytest.fixture(scope="module")
def mc_whole():
    p = _plan(MC, "whole")
    yield p
    p.close()


@pytest.fixture(scope="module")
def pair_whole():
    p = _plan(PAIR, "whole")
    yield p
    p.close()


def _run(p, ta, tb, M, N, acc="f32", reps=1):
    outs = []
    for _ in range(reps):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        p.run(ta, tb, c, acc=acc)
        outs.append(c)
    p.check_error()
    return outs


@pytest.mark.parametrize("acc", ["f32", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bitwise_equal_to_one_pair_kernel(mc_whole, pair_whole, shape, acc):
    M, N, K = shape
    a, b = wl.draw(M, N, K, seed=7 * M + N + K)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref = _run(pair_whole, ta, tb, M, N, acc)[0]
    got = _run(mc_whole, ta, tb, M, N, acc)[0]
    assert torch.equal(got, ref), f"{shape} {acc}: differs from the one-pair kernel"
    if M * N * K <= 3000 * 5000 * 4104:
        assert_close(got.cpu().numpy(), oracle.gemm_f64(a, b), acc, f"{shape} {acc}")


def test_repeated_launches_agree_bit_for_bit(mc_whole, pair_whole):
    """40 back-to-back launches of the ragged workload (programmatic dependent
    launch on, so consecutive kernels overlap) against the one-pair result."""
    M, N, K = 3000, 5000, 4104
    a, b = wl.draw(M, N, K, seed=3)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref = _run(pair_whole, ta, tb, M, N)[0]
    for i, c in enumerate(_run(mc_whole, ta, tb, M, N, reps=40)):
        assert torch.equal(c, ref), f"launch {i} differs"


@pytest.mark.parametrize("layouts", ["kn", "mk", "mn"])
def test_mn_contiguous_operands_bitwise(layouts):
    """M/N-contiguous A is loaded as two 64-wide boxes per CTA; with multicast
    each pair loads one of them."""
    M, N, K = 1000, 1280, 776
    a, b = wl.draw(M, N, K, seed=99)
    la = g.MN_CONTIGUOUS if layouts[0] == "m" else g.K_CONTIGUOUS
    lb = g.MN_CONTIGUOUS if layouts[1] == "n" else g.K_CONTIGUOUS
    ta = torch.from_numpy(a if la == g.K_CONTIGUOUS else np.ascontiguousarray(a.T)).cuda()
    tb = torch.from_numpy(b if lb == g.K_CONTIGUOUS else np.ascontiguousarray(b.T)).cuda()
    outs = []
    for v in (PAIR, MC):
        p = _plan(v, "whole")
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        p.run_ex_ptr(ta.data_ptr(), la, tb.data_ptr(), lb, c.data_ptr(), M, N, K, "f32",
                     torch.cuda.current_stream().cuda_stream)
        p.check_error()
        p.close()
        outs.append(c)
    assert torch.equal(outs[0], outs[1]), layouts
    assert_close(outs[1].cpu().numpy(), oracle.gemm_f64(a, b), "f32", layouts)


def test_automatic_choice(plan):
    """Chosen for K-contiguous rows whose pitch is not a multiple of 128 bytes
    (the ragged workload), not for aligned rows or M/N-contiguous operands."""
    assert plan.describe(3000, 5000, 4104)["variant"] == MC
    assert plan.describe(8192, 8192, 8200)["variant"] == MC
    assert plan.describe(8192, 8192, 8192)["variant"] == PAIR
    assert plan.describe(4096, 4096, 4096)["variant"] == PAIR
    M, N, K = 1000, 1280, 1032
    a, b = wl.draw(M, N, K, seed=98)
    assert plan.describe(M, N, K)["variant"] == MC
    c = _run(plan, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), M, N)[0]
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", "auto")


def test_describe_reports_two_pair_clusters():
    p = _plan(MC, "auto")
    d = p.describe(3000, 5000, 4104)
    units = p.resident_units()
    p.close()
    assert d["variant"] == MC
    assert d["grid_ctas"] == 4 * d["units"] and 1 <= d["units"] <= units["quads"]
    assert g.variant_info(MC) == {"ctas": 4, "tile_m": 256, "tile_n": 512, "swap": False}
