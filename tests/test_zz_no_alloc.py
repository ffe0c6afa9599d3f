"""The allocation-free entry point, gemm_run_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory: code running under
an allocator that owns every byte of the GPU (a framework's caching allocator
or a fixed arena), and latency-bound loops that cannot take cudaMalloc's
implicit device synchronisation.  Such callers cannot create a plan (that
allocates the kernel's watchdog record), so this entry point keeps that
record in a static device array inside the library.

Checked here: on two calls in a row (the second reuses the array the first
one left behind) its output matches the CPU oracle element by element within
the tolerance the other GPU tests use, and stays within that tolerance of
gemm_run's output (the two may pick different tile shapes, so they need not
agree bit for bit); K == 0 writes zeros over whatever C held; it rejects bad
arguments like gemm_run, including pointers that are not memory of the
current device.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp16_gemm_04_gb300 as g
import gemm_workloads as wl
import oracle
from conftest import assert_close

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
def test_noalloc_matches_the_oracle_on_two_calls(noalloc, plan, acc):
    M, N, K = 1000, 776, 4104          # several tiles, ragged M, N and K tails
    a, b = wl.draw(M, N, K, seed=41)
    ref = oracle.gemm_f64(a, b)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    via_plan = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    plan.run(ta, tb, via_plan, acc=acc)
    plan.check_error()
    via_plan = via_plan.cpu().numpy().astype(np.float64)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        status = noalloc(ta.data_ptr(), tb.data_ptr(), c.data_ptr(), M, N, K, ACC[acc], stream)
        assert status == 0, f"call {call}: {g.status_string(status)}"
        torch.cuda.synchronize()
        got = c.cpu().numpy()
        assert_close(got, ref, acc, f"gemm_run_noalloc call {call}")
        assert_close(got, via_plan, acc, f"gemm_run_noalloc call {call} vs gemm_run")


def test_noalloc_k0_writes_zeros(noalloc):
    M, N = 300, 136
    a = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((N, 0), dtype=torch.float16, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, 0, 0, s) == 0
    torch.cuda.synchronize()
    assert bool((c == 0).all())


def test_noalloc_rejects_bad_arguments(noalloc):
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    c = torch.full((64, 64), 3.0, dtype=torch.float16, device="cuda")
    h = torch.ones((64, 64), dtype=torch.float16).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    assert noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 60, 0, s) == 2   # K % 8
    assert noalloc(a.data_ptr() + 2, a.data_ptr(), c.data_ptr(), 64, 64, 64, 0, s) == 2
    assert noalloc(a.data_ptr(), a.data_ptr(), None, 64, 64, 64, 0, s) == 1
    assert noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 64, 5, s) == 1
    # host memory, pinned or not, is not memory of the current device
    assert noalloc(h.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 64, 0, s) == 1
    assert noalloc(a.data_ptr(), a.data_ptr(), h.data_ptr(), 64, 64, 64, 0, s) == 1
    hn = np.ones((64, 64), dtype=np.float16)
    assert noalloc(a.data_ptr(), hn.ctypes.data, c.data_ptr(), 64, 64, 64, 0, s) == 1
    torch.cuda.synchronize()
    assert bool((c == 3.0).all())
