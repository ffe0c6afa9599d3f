"""Split-K clusters (tc_swap_{16,32,64}x128_k2, tc_single_128x64_k4): the CTAs
of a cluster share every tile they are given, each accumulating its own
k-slice.  In tc_single_128x64_k4 the CTAs of rank > 0 write their fp32
partial tiles into the shared memory of rank 0, which adds them to its own in
rank order and stores C; in the swapped-roles pairs each CTA finishes half of
the tile's rows of C and receives the other CTA's partial of them.

Checked here against the CPU oracle: k-slices of unequal length (the number
of k-blocks not a multiple of the cluster size), one k-block per CTA, ragged
M, N and K, more tiles than resident clusters (each cluster then takes
several tiles in turn, so a partial slot must be freed before the next
tile's partial may land in it), results identical from run to run, the
automatic choice of these variants, and fp16 accumulation falling back to
whole tiles."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import VARIANTS_SPLITK, assert_close

pytestmark = pytest.mark.gpu

SWAP_K2 = ["tc_swap_16x128_k2", "tc_swap_32x128_k2", "tc_swap_64x128_k2"]
K4 = "tc_single_128x64_k4"
BASE = {"tc_swap_16x128_k2": "tc_swap_16x128_s11", "tc_swap_32x128_k2": "tc_swap_32x128_s10",
        "tc_swap_64x128_k2": "tc_swap_64x128_s8", K4: "tc_single_128x64_s8"}


def _plan(variant):
    p = g.Plan(0)
    p.set_variant(variant)
    return p


def _gemm(p, a, b, acc="f32", reps=1):
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    outs = []
    for _ in range(reps):
        c = torch.full((a.shape[0], b.shape[0]), float("nan"), dtype=torch.float16, device="cuda")
        p.run(ta, tb, c, acc=acc)
        outs.append(c)
    p.check_error()
    return [c.cpu().numpy() for c in outs]


# (M, N, K): k-blocks 5 (slices 2/3 or 1/1/1/2), 4 (one per CTA of a k4
# cluster), 2 (one per CTA of a k2 cluster), 130 with a ragged last block.
SHAPES = [(40, 392, 320), (100, 520, 256), (64, 1032, 128), (16, 2056, 8264), (200, 136, 1032)]


@pytest.mark.parametrize("variant", VARIANTS_SPLITK)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_matches_oracle(variant, shape):
    M, N, K = shape
    a, b = wl.draw(M, N, K, seed=M + 3 * N + 7 * K)
    p = _plan(variant)
    d = p.describe(M, N, K)
    got = _gemm(p, a, b)[0]
    p.close()
    slices = 4 if variant == K4 else 2
    if (K + 63) // 64 >= slices:
        assert d["variant"] == variant
    else:                      # fewer k-blocks than CTAs: whole tiles instead
        assert d["variant"] == BASE[variant]
    assert_close(got, oracle.gemm_f64(a, b), "f32", f"{variant} {shape}")


@pytest.mark.parametrize("variant", VARIANTS_SPLITK)
def test_more_tiles_than_clusters(variant):
    """Every cluster takes several tiles in turn: each partial slot is
    reused from tile to tile."""
    p = _plan(variant)
    units = p.resident_units()
    M, N, K = (2048, 2048, 512) if variant == K4 else (64, 65536, 256)
    d = p.describe(M, N, K)
    assert d["variant"] == variant and d["dp_tiles"] > 2 * d["units"], d
    a, b = wl.draw(M, N, K, seed=61)
    outs = _gemm(p, a, b, reps=3)
    p.close()
    assert_close(outs[0], oracle.gemm_f64(a, b), "f32", variant)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16)), "runs differ"
    assert units["ctas"] >= d["grid_ctas"]


def test_automatic_choice(plan):
    assert plan.describe(64, 8192, 8192)["variant"] == "tc_swap_64x128_k2"
    assert plan.describe(32, 8192, 8192)["variant"] == "tc_swap_32x128_k2"
    assert plan.describe(16, 8192, 8192)["variant"] == "tc_swap_16x128_k2"
    d = plan.describe(256, 256, 4096)       # 8 tiles, 16 k-blocks per CTA
    assert d["variant"] == K4 and d["grid_ctas"] == 4 * 8 and d["sk_units"] == 0
    assert plan.describe(128, 1024, 8192)["variant"] == K4
    # 512^3: 2 k-blocks per CTA, whole tiles are faster
    assert plan.describe(512, 512, 512)["variant"] == "tc_single_128x64_s8"
    # many tiles: whole tiles per CTA as before
    assert plan.describe(16, 16384, 16384)["variant"] == "tc_swap_16x128_s11"
    assert plan.describe(4096, 4096, 4096)["variant"] == "tc_pair_256x256_s6"
    # too few k-blocks for four slices
    assert plan.describe(512, 512, 192)["variant"] == "tc_single_128x64_s8"
    # fp16 accumulation keeps whole tiles
    assert plan.describe(512, 512, 512, acc="f16")["variant"] == "tc_single_128x64_s8"
    assert plan.describe(64, 8192, 8192, acc="f16")["variant"] == "tc_swap_64x128_s8"


@pytest.mark.parametrize("shape", [(256, 256, 4096), (128, 1024, 8192), (64, 8192, 8192),
                                   (16, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_automatic_shapes_match_the_oracle(plan, shape):
    M, N, K = shape
    a, b = wl.draw(M, N, K, seed=62)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    plan.run(ta, tb, c)
    plan.check_error()
    if M * N <= 128 * 1024:
        assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), "f32", str(shape))
    else:
        cols = wl.sample_indices(N, 256, 63)
        assert_close(c.cpu().numpy()[:, cols], oracle.gemm_f64(a, b[cols]), "f32", str(shape))


@pytest.mark.parametrize("variant", VARIANTS_SPLITK)
def test_fp16_accumulation_falls_back_to_whole_tiles(variant):
    p = _plan(variant)
    M, N, K = 64, 1032, 512
    d = p.describe(M, N, K, acc="f16")
    a, b = wl.draw(M, N, K, seed=64)
    got = _gemm(p, a, b, acc="f16")[0]
    p.close()
    assert d["variant"] != variant and not d["variant"].endswith(("_k2", "_k4"))
    assert_close(got, oracle.gemm_f64(a, b), "f16", variant)
