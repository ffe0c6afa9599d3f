"""The allocation-free entry point, gemm_run_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory: code running under
an allocator that owns every byte of the GPU (a framework's caching allocator
or a fixed arena), and latency-bound loops that cannot take cudaMalloc's
implicit device synchronisation.  Such callers cannot create a plan (that
allocates the kernel's watchdog record), so this entry point keeps that
record in a static device array inside the library.

Checked here: its output matches gemm_run's within the tolerance the other
GPU tests use, on two calls in a row (the second call reuses the array the
first one left behind), and it rejects bad arguments like gemm_run.  This file
sorts last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
from conftest import TOL, error_stats

pytestmark = pytest.mark.gpu

ACC = {"f32": 0, "f16": 1}


@pytest.fixture(scope="module")
def noalloc():
    g.build()
    lib = ctypes.CDLL(g.LIB_PATH)
    fn = lib.gemm_run_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    return fn


@pytest.mark.parametrize("acc", ["f32", "f16"])
def test_noalloc_matches_gemm_run_on_two_calls(noalloc, plan, acc):
    M, N, K = 1000, 776, 4104          # several tiles, ragged M, N and K tails
    a, b = wl.draw(M, N, K, seed=41)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    plan.run(ta, tb, ref, acc=acc)
    plan.check_error()
    ref_np = ref.cpu().numpy().astype(np.float64)
    stream = torch.cuda.current_stream().cuda_stream
    atol = TOL[acc][0]
    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        status = noalloc(ta.data_ptr(), tb.data_ptr(), c.data_ptr(), M, N, K, ACC[acc], stream)
        assert status == 0, f"call {call}: {g.status_string(status)}"
        torch.cuda.synchronize()
        st = error_stats(c.cpu().numpy(), ref_np)
        assert st["finite"], f"call {call}: unwritten or non-finite outputs"
        assert st["max_abs"] <= atol, f"call {call}: max |diff| {st['max_abs']} > {atol}"


def test_noalloc_rejects_bad_arguments(noalloc):
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    c = torch.full((64, 64), 3.0, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 60, 0, s) == 2   # K % 8
    assert noalloc(a.data_ptr() + 2, a.data_ptr(), c.data_ptr(), 64, 64, 64, 0, s) == 2
    assert noalloc(a.data_ptr(), a.data_ptr(), None, 64, 64, 64, 0, s) == 1
    assert noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 64, 5, s) == 1
    torch.cuda.synchronize()
    assert bool((c == 3.0).all())
