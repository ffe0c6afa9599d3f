"""The kernel's watchdog, exercised without faulting the GPU: the producer is
told to skip one k-block's load and never declare its bytes, so the MMA
issuer's wait for that stage can only end by timing out.  The kernel must
record GEMM_ERR_TIMEOUT, leave every loop, free tensor memory and return;
the host reads the status, and the next normal call must succeed."""
import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import VARIANTS, assert_close

pytestmark = pytest.mark.gpu

TIMEOUT_NS = 50_000_000    # 50 ms for any single wait in the injected run
# The first wait to give up is the MMA issuer's wait for the skipped stage
# (site 2) or, racing it by microseconds, the epilogue's wait for that tile's
# accumulator (site 4); both are the stuck tile's own waits.
STUCK_SITES = (2, 4)


@pytest.mark.parametrize("variant", VARIANTS)
def test_stuck_wait_reports_timeout_and_context_survives(variant):
    p = g.Plan(0)
    p.set_variant(variant)
    M, N, K = 1024, 1024, 1024
    a, b = wl.draw(M, N, K, seed=51)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()

    # Unit 0's first piece of work: the first shared tile when the schedule
    # has a stream-K share (it runs first), else tile 0.
    d = p.describe(M, N, K)
    first_tile = d["dp_tiles"] if d["sk_units"] > 0 else 0
    p.set_watchdog(timeout_ns=TIMEOUT_NS, skip_k_block=0)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    p.run(ta, tb, c)                          # the launch itself succeeds
    status = p.check_error_status()
    assert status == 5, g.status_string(status)
    code, site, cta, tile = p.last_error_detail()
    # The stuck stage belongs to unit 0: CTA 0 or another CTA of its cluster
    # (a pair, or two pairs sharing A, where both pairs wait for it).
    assert code == 5 and site in STUCK_SITES and 0 <= cta < 4 and tile == first_tile
    assert p.check_error_status() == 0        # the record was cleared

    # Back to normal: same plan, same context.
    p.set_watchdog(0, -1)
    c2 = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    p.run(ta, tb, c2)
    p.check_error()
    assert_close(c2.cpu().numpy(), oracle.gemm_f64(a, b), "f32", f"after timeout {variant}")
    p.close()


def test_watchdog_arguments_are_checked(plan):
    with pytest.raises(g.GemmError):
        plan.set_watchdog(0, -2)
