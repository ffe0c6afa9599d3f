"""Swapped-roles epilogue (the tc_swap_* variants, whole tiles and split-K
pairs).  A thread holds one column of C and that column's values down the
tile's rows; each group of eight lanes transposes 8 x 8 blocks in registers
and writes eight columns of one row as a 16-byte store, skipping rows at or
past M and column groups at or past N.  In a split-K pair each CTA finishes
half of the tile's rows and receives the other CTA's partial of them.

Checked against the CPU oracle for row counts inside, at the edges of and
past each 8-row block and each half tile, with N not a multiple of the
128-column tile (the last tile holds one group of eight columns), and with C
between two runs of sentinels that must stay untouched."""
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import VARIANTS, assert_close

pytestmark = pytest.mark.gpu

SWAPPED = [v for v in VARIANTS if v.startswith("tc_swap_")]
# 1..64 rows: inside the first block, on block edges, one past them, inside
# the second half of a 16-, 32- or 64-row split tile, a full tile.
ROWS = [1, 5, 8, 9, 15, 16, 17, 24, 31, 33, 40, 47, 57, 63, 64]
N, K = 392, 320        # 3 tiles of 128 columns + 8; 5 k-blocks (split 2 / 3)
GUARD = 4096


@pytest.fixture(scope="module")
def plans():
    ps = {}
    for v in SWAPPED:
        p = g.Plan(0)
        p.set_variant(v)
        ps[v] = p
    yield ps
    for p in ps.values():
        p.close()


@pytest.mark.parametrize("M", ROWS)
@pytest.mark.parametrize("variant", SWAPPED)
def test_rows_and_column_groups(plans, variant, M):
    p = plans[variant]
    assert p.describe(M, N, K)["variant"] == variant
    a, b = wl.draw(M, N, K, seed=1000 + M)
    buf = torch.full((GUARD + M * N + GUARD,), 1234.0, dtype=torch.float16, device="cuda")
    c = buf[GUARD:GUARD + M * N].view(M, N)
    c.fill_(float("nan"))
    p.run(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), c)
    p.check_error()
    host = buf.cpu()
    assert bool((host[:GUARD] == 1234.0).all()), "write before C"
    assert bool((host[GUARD + M * N:] == 1234.0).all()), "write after C"
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", f"{variant} M={M}")


WHOLE = {"tc_swap_16x128_k2": "tc_swap_16x128_s11", "tc_swap_32x128_k2": "tc_swap_32x128_s10",
         "tc_swap_64x128_k2": "tc_swap_64x128_s8"}


@pytest.mark.parametrize("variant", sorted(WHOLE))
def test_long_k_split_and_whole(plans, variant):
    """K = 4104 (65 k-blocks, the last one ragged): the split pair and the
    whole-tile variant both match the oracle, and the split pair's result is
    identical from run to run."""
    M = int(variant.split("_")[2].split("x")[0])
    Kl = 4104
    a, b = wl.draw(M, N, Kl, seed=77)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref = oracle.gemm_f64(a, b)
    outs = []
    for _ in range(3):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        plans[variant].run(ta, tb, c)
        outs.append(c)
    plans[variant].check_error()
    cw = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    plans[WHOLE[variant]].run(ta, tb, cw)
    plans[WHOLE[variant]].check_error()
    for c in outs[1:]:
        assert torch.equal(c, outs[0]), "split result changed between runs"
    assert_close(outs[0].cpu().numpy(), ref, "f32", f"{variant} split")
    assert_close(cw.cpu().numpy(), ref, "f32", f"{WHOLE[variant]} whole")
