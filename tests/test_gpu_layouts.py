"""M/N-contiguous operands (gemm_run_ex): A stored [K, M] and/or B stored
[K, N] against the oracle on the same logical matrices, on every variant
that takes them, plus exact closed forms that expose a wrong descriptor
stride or a transposed operand."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import VARIANTS_WIDE, assert_close

pytestmark = pytest.mark.gpu

LAYOUTS = [(g.K_CONTIGUOUS, g.MN_CONTIGUOUS), (g.MN_CONTIGUOUS, g.K_CONTIGUOUS),
           (g.MN_CONTIGUOUS, g.MN_CONTIGUOUS)]
LAYOUT_IDS = ["A_k-B_n", "A_m-B_k", "A_m-B_n"]


def stored(x, layout):
    """Device copy of logical matrix x ([rows, K]) in the given storage."""
    if layout == g.K_CONTIGUOUS:
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x.T)).cuda()   # [K, rows]


def run_ex(plan, a, la, b, lb, acc="f32"):
    M, K = a.shape
    N = b.shape[0]
    ta, tb = stored(a, la), stored(b, lb)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    plan.run_ex_ptr(ta.data_ptr(), la, tb.data_ptr(), lb, c.data_ptr(), M, N, K, acc,
                    torch.cuda.current_stream().cuda_stream)
    plan.check_error()
    return c.cpu().numpy()


@pytest.mark.parametrize("variant", VARIANTS_WIDE)
@pytest.mark.parametrize("layouts", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("shape", [(256, 512, 384), (296, 520, 328), (136, 1032, 1000),
                                   (64, 264, 72), (1024, 776, 4104)],
                         ids=lambda s: "x".join(map(str, s)))
def test_layouts_match_oracle(plans, variant, layouts, shape):
    M, N, K = shape
    a, b = wl.draw(M, N, K, seed=M + N + K)
    got = run_ex(plans[variant], a, layouts[0], b, layouts[1])
    assert_close(got, oracle.gemm_f64(a, b), "f32", f"{shape} {variant} {layouts}")


@pytest.mark.parametrize("layouts", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("acc", ["f32", "f16"])
def test_layouts_auto_and_f16(plan, layouts, acc):
    for shape in [(8, 8, 64), (40, 264, 136), (520, 264, 1032)]:
        M, N, K = shape
        a, b = wl.draw(M, N, K, seed=7 * M + N)
        assert_close(run_ex(plan, a, layouts[0], b, layouts[1], acc), oracle.gemm_f64(a, b),
                     acc, f"{shape} {layouts}")


@pytest.mark.parametrize("variant", VARIANTS_WIDE)
@pytest.mark.parametrize("layouts", LAYOUTS, ids=LAYOUT_IDS)
def test_layouts_identity_and_permutation_exact(plans, variant, layouts):
    K = 256
    _, b = wl.draw(K, 264, K, seed=91)
    c = run_ex(plans[variant], wl.identity(K), layouts[0], b, layouts[1])
    assert np.array_equal(c.view(np.uint16), np.ascontiguousarray(b.T).view(np.uint16))
    a, _ = wl.draw(192, 256, 512, seed=92)
    p, perm = wl.permutation(256, 512, seed=93)
    c = run_ex(plans[variant], a, layouts[0], p, layouts[1])
    assert np.array_equal(c.view(np.uint16), np.ascontiguousarray(a[:, perm]).view(np.uint16))


def test_torch_views_pick_the_layout(plan):
    """gemm(x, w.t()) with w stored [K, N] computes x @ w without a copy."""
    M, N, K = 264, 520, 200
    x, wt = wl.draw(M, N, K, seed=94)         # wt is logical B = w.T, [N, K]
    w = torch.from_numpy(np.ascontiguousarray(wt.T)).cuda()    # stored [K, N]
    c = g.gemm(torch.from_numpy(x).cuda(), w.t(), plan=plan)
    torch.cuda.synchronize()
    assert_close(c.cpu().numpy(), oracle.gemm_f64(x, wt), "f32", "x @ w")


def test_layout_rules(plan):
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    c = torch.zeros((60, 64), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    lib = g.load()
    # A stored [K, M] with M = 60: rows of A not 16-byte aligned
    assert lib.gemm_run_ex(plan.handle, a.data_ptr(), 1, a.data_ptr(), 0, c.data_ptr(),
                           60, 64, 64, 0, s) == 2
    # K need not be a multiple of 8 when both operands are M/N-contiguous
    a2 = torch.ones((12, 64), dtype=torch.float16, device="cuda")     # [K=12, M=64]
    b2 = torch.ones((12, 64), dtype=torch.float16, device="cuda")     # [K=12, N=64]
    c2 = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    assert lib.gemm_run_ex(plan.handle, a2.data_ptr(), 1, b2.data_ptr(), 1, c2.data_ptr(),
                           64, 64, 12, 0, s) == 0
    plan.check_error()
    assert bool((c2 == 12.0).all())
    assert lib.gemm_run_ex(plan.handle, a.data_ptr(), 2, a.data_ptr(), 0, c.data_ptr(),
                           64, 64, 64, 0, s) == 1
