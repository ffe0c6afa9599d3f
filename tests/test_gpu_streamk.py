"""The stream-K tail against the oracle: the last tiles' k-blocks are shared
between units, each unit parks an fp32 partial tile in the plan's workspace,
and the last contributor sums the partials in unit order and stores the
tile.  Forced on for small shapes (many shared tiles, several contributors
per tile), and checked as chosen automatically on the full workloads."""
import numpy as np
import pytest
import torch

import gemm_workloads as wl
import oracle
from conftest import VARIANTS, assert_close, run_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(300, 520, 328), (129, 264, 1032), (1000, 776, 4104), (640, 1280, 64),
          (2000, 40, 256), (257, 520, 520), (8, 8, 4096), (3000, 5000, 512)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forced_streamk_matches_oracle(plans_streamk, variant, shape):
    p = plans_streamk[variant]
    M, N, K = shape
    d = p.describe(M, N, K)
    a, b = wl.draw(M, N, K, seed=M + 3 * N + 7 * K)
    c = run_gpu(p, a, b, "f32")
    assert_close(c, oracle.gemm_f64(a, b), "f32", f"{shape} {variant} {d}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_streamk_is_deterministic(plans_streamk, variant):
    """Partials are summed in unit order, so repeated runs agree bit for bit."""
    p = plans_streamk[variant]
    M, N, K = 1000, 776, 4104
    a, b = wl.draw(M, N, K, seed=61)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    outs = []
    for _ in range(5):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        p.run(ta, tb, c)
        outs.append(c)
    p.check_error()
    for c in outs[1:]:
        assert torch.equal(c, outs[0])


def test_streamk_counters_reset_between_calls(plans_streamk):
    """The tail counters are left at zero by each launch: alternate shapes with
    different tails, many times, on one plan."""
    p = plans_streamk[VARIANTS[0]]
    cases = []
    for shape in [(300, 520, 328), (640, 1280, 64), (1000, 776, 4104)]:
        a, b = wl.draw(*shape, seed=sum(shape))
        cases.append((shape, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                      oracle.gemm_f64(a, b)))
    for it in range(4):
        for shape, ta, tb, ref in cases:
            c = torch.full(shape[:2], float("nan"), dtype=torch.float16, device="cuda")
            p.run(ta, tb, c)
            p.check_error()
            assert_close(c.cpu().numpy(), ref, "f32", f"{shape} round {it}")


def test_auto_schedule_uses_the_tail_on_quantized_waves(plan):
    d = plan.describe(4096, 4096, 4096)
    assert d["sk_units"] > 0 and d["dp_tiles"] % d["units"] == 0
    d = plan.describe(16384, 16384, 16384)
    assert d["sk_units"] == 0           # 53.9 waves: the tail would not pay
    d = plan.describe(8192, 8192, 8192, "f16")
    assert d["sk_units"] == 0           # fp16 accumulation keeps whole tiles
    d = plan.describe(512, 512, 512)
    assert d["sk_units"] == 0           # fewer tiles than units: whole tiles
    d = plan.describe(1024, 8192, 8192)
    assert d["sk_units"] > 0 and d["dp_tiles"] == d["units"]   # only the last wave is shared


def test_auto_schedule_swapped_roles(plan):
    """Few tall tiles (C with at most 64 rows): each tile is cut into the
    same whole number of k-pieces when its partial tiles are large or there
    are pieces to spare, else the units' ranges run on across tiles.  Two
    pieces per tile run as split-K clusters of two CTAs (the partial goes
    through shared memory); more pieces through the stream-K share."""
    d = plan.describe(64, 8192, 8192)         # 64 tiles of 128 columns: 2 pieces each
    assert d["variant"] == "tc_swap_64x128_k2" and d["sk_units"] == 0
    assert d["units"] == 64 and d["grid_ctas"] == 128 and d["dp_tiles"] == 64
    d = plan.describe(16, 8192, 8192)         # 2 x 64 tiles <= 152 units: 2 pieces each
    assert d["variant"] == "tc_swap_16x128_k2" and d["grid_ctas"] == 128
    d = plan.describe(64, 4096, 8192)         # 32 tiles: 4 pieces each, stream-K share
    assert d["variant"] == "tc_swap_64x128_s8" and d["sk_units"] == 128
    d = plan.describe(48, 12288, 8192)        # 96 tiles, one piece each: whole tiles
    assert d["sk_units"] == 0 and d["units"] == 96 and d["dp_tiles"] == 96
    d = plan.describe(16, 16384, 16384)       # 128 tiles of 16 rows: ranges over all units
    assert d["sk_units"] == d["units"] and d["sk_iters"] == 128 * 256


def test_every_share_unit_has_work():
    """The fix-up counts on every unit of a stream-K share contributing: no
    schedule may give a unit of the share an empty k-range.  Checked on the
    host-side layout (no launch) for every variant and schedule mode over a
    sweep of shapes, tiny K and few tiles included."""
    import dense_fp16_gemm_04_gb300 as g
    shapes = [(8, 120, 264), (16, 128, 64), (64, 8192, 1024), (64, 8192, 8192), (16, 8192, 8192),
              (48, 12288, 8192), (16, 16384, 16384), (300, 520, 328), (1000, 776, 4104),
              (4096, 4096, 1024), (4096, 4096, 4096), (3000, 5000, 4104), (129, 264, 1032),
              (8, 8, 4096), (2000, 40, 256), (16, 1024, 65536), (256, 256, 8)]
    for variant in g.variant_names():
        for mode in ("auto", "streamk"):
            p = g.Plan(0)
            p.set_variant(variant)
            p.set_schedule(mode)
            for M, N, K in shapes:
                d = p.describe(M, N, K)
                if d["sk_units"]:
                    floor = 1 if mode == "streamk" else 16
                    assert d["sk_iters"] >= floor * d["sk_units"], (variant, mode, (M, N, K), d)
            p.close()
