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
