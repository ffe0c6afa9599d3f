import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def read_golden(name):
    """Parse a tests/golden fixture: '# comment' lines, then 'NAME rows cols'
    headers followed by that many rows of numbers, or 'key value' pairs."""
    path = os.path.join(ROOT, "tests", "golden", name)
    mats, scalars = {}, {}
    with open(path) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
    i = 0
    while i < len(lines):
        parts = lines[i].split()
        if len(parts) == 3 and parts[1].isdigit() and parts[2].isdigit():
            r, c = int(parts[1]), int(parts[2])
            rows = [[float(v) for v in lines[i + 1 + t].split()] for t in range(r)]
            assert all(len(row) == c for row in rows)
            mats[parts[0]] = rows
            i += 1 + r
        else:
            scalars[parts[0]] = float(parts[1])
            i += 1
    return mats, scalars


# ------------------------------------------------------------ GPU helpers --
# Pass bounds on unit-variance outputs: fp32 accumulation |err| <= 1e-2 and
# |err| / max(|ref|, 1) <= 1e-2; native fp16 accumulation |err| <= 5e-2 (the
# bound tilus "Four Consumers, FP16 Accumulation, and a TMA Epilogue" uses for
# its K=8192 fp16-accumulated check, "The Register Budget Problem").
TOL = {"f32": (1e-2, 1e-2), "f16": (5e-2, None)}


def error_stats(got, ref):
    import numpy as np
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), 1.0)
    return {"max_abs": float(err.max()) if err.size else 0.0,
            "mean_abs": float(err.mean()) if err.size else 0.0,
            "p99_abs": float(np.percentile(err, 99)) if err.size else 0.0,
            "max_rel": float(rel.max()) if rel.size else 0.0,
            "finite": bool(np.isfinite(got).all())}


def assert_close(got, ref, acc, what=""):
    st = error_stats(got, ref)
    atol, rtol = TOL[acc]
    assert st["finite"], f"{what}: non-finite outputs"
    assert st["max_abs"] <= atol, f"{what}: max |err| {st['max_abs']:.4g} > {atol} ({st})"
    if rtol is not None:
        assert st["max_rel"] <= rtol, f"{what}: max rel err {st['max_rel']:.4g} > {rtol}"
    return st


# Kernel variants of the library, in its table order (checked against the
# library by test_abi_host.py::test_variant_table).
VARIANTS = ["tc_pair_256x256_s6", "tc_single_128x256_s4", "tc_pair_256x128_s8",
            "tc_single_128x64_s8", "tc_swap_16x128_s11", "tc_swap_32x128_s10",
            "tc_swap_64x128_s8", "tc_pair_mc_256x256_s6", "tc_swap_16x128_k2",
            "tc_swap_32x128_k2", "tc_swap_64x128_k2", "tc_single_128x64_k4"]
# The variants built for large M (the swapped-roles ones, made for a few rows
# of C, would take minutes on the full-size squares).
VARIANTS_WIDE = [v for v in VARIANTS if "swap" not in v]
# Split-K clusters: the CTAs of a cluster share each tile, one k-slice each.
VARIANTS_SPLITK = [v for v in VARIANTS if v.endswith(("_k2", "_k4"))]


@pytest.fixture(scope="session")
def plan():
    """A plan with automatic variant choice."""
    import dense_fp16_gemm_04_gb300 as g
    g.build()
    p = g.Plan(0)
    yield p
    p.close()


@pytest.fixture(scope="session")
def plans_streamk():
    """One plan per kernel variant, forced to use the stream-K tail whenever
    the shape allows it."""
    import dense_fp16_gemm_04_gb300 as g
    g.build()
    ps = {}
    for name in VARIANTS:
        ps[name] = g.Plan(0)
        ps[name].set_variant(name)
        ps[name].set_schedule("streamk")
    yield ps
    for p in ps.values():
        p.close()


@pytest.fixture(scope="session")
def plans():
    """One plan per kernel variant, each forced to that variant."""
    import dense_fp16_gemm_04_gb300 as g
    g.build()
    ps = {}
    for name in VARIANTS:
        ps[name] = g.Plan(0)
        ps[name].set_variant(name)
    yield ps
    for p in ps.values():
        p.close()


def to_dev(x):
    import torch
    return torch.from_numpy(x).cuda()


def run_gpu(plan, a, b, acc="f32", fill=float("nan")):
    """C = A @ B.T on the GPU through the C ABI; C is pre-filled with NaN so
    any element the kernel fails to write shows up."""
    import numpy as np
    import torch
    ta, tb = to_dev(a), to_dev(b)
    c = torch.full((a.shape[0], b.shape[0]), fill, dtype=torch.float16, device="cuda")
    plan.run(ta, tb, c, acc=acc)
    plan.check_error()
    return c.cpu().numpy()
