"""Seeded random cases over the whole configuration space — shape (ragged
edges included), kernel variant, operand layouts, accumulation and work
schedule — each checked against the oracle on every element."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import VARIANTS, assert_close

pytestmark = pytest.mark.gpu

SWAPPED = {"tc_swap_16x128_s11", "tc_swap_32x128_s10", "tc_swap_64x128_s8"}


def cases(n=150, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        variant = VARIANTS[rng.integers(len(VARIANTS))]
        M = int(rng.integers(1, 97 if variant in SWAPPED else 700))
        N = 8 * int(rng.integers(1, 90))
        K = 8 * int(rng.integers(1, 180))
        la = g.K_CONTIGUOUS if variant in SWAPPED or rng.random() < 0.5 else g.MN_CONTIGUOUS
        lb = g.K_CONTIGUOUS if variant in SWAPPED or rng.random() < 0.5 else g.MN_CONTIGUOUS
        if la == g.MN_CONTIGUOUS:
            M = max(8, M - M % 8)
        acc = "f16" if rng.random() < 0.3 else "f32"
        sched = ["auto", "whole", "streamk"][int(rng.integers(3))]
        out.append((variant, M, N, K, la, lb, acc, sched, int(rng.integers(1 << 30))))
    return out


@pytest.fixture(scope="module")
def fuzz_plans():
    ps = {}
    for v in VARIANTS:
        for s in ("auto", "whole", "streamk"):
            p = g.Plan(0)
            p.set_variant(v)
            p.set_schedule(s)
            ps[(v, s)] = p
    yield ps
    for p in ps.values():
        p.close()


@pytest.mark.parametrize("case", cases(), ids=lambda c: f"{c[0][3:]}-{c[1]}x{c[2]}x{c[3]}-"
                         f"{'km'[c[4]]}{'kn'[c[5]]}-{c[6]}-{c[7]}")
def test_fuzz(fuzz_plans, case):
    variant, M, N, K, la, lb, acc, sched, seed = case
    p = fuzz_plans[(variant, sched)]
    a, b = wl.draw(M, N, K, seed=seed % 100000)
    ta = torch.from_numpy(a if la == g.K_CONTIGUOUS else np.ascontiguousarray(a.T)).cuda()
    tb = torch.from_numpy(b if lb == g.K_CONTIGUOUS else np.ascontiguousarray(b.T)).cuda()
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    p.run_ex_ptr(ta.data_ptr(), la, tb.data_ptr(), lb, c.data_ptr(), M, N, K, acc,
                 torch.cuda.current_stream().cuda_stream)
    p.check_error()
    assert_close(c.cpu().numpy(), oracle.gemm_f64(a, b), acc, f"{case} {p.describe(M, N, K, acc)}")
