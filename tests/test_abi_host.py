"""Host-only checks of the C ABI: the library loads without a GPU, exports
every entry point include/gemm.h declares, and its host-side answers (status
names, variant table, argument rejection) are right.  No kernel is launched."""
import ctypes
import os
import re

import pytest

import dense_fp16_gemm_04_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gemm.h")).read()
    return re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    g.build()
    return g.load()


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"gemm_plan_create", "gemm_run", "gemm_plan_destroy"} <= names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(g.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_no_torch_types_in_the_header():
    src = open(os.path.join(ROOT, "include", "gemm.h")).read()
    assert "torch" not in src.lower().replace("pytorch", "")
    assert "at::" not in src and "c10" not in src


def test_status_strings(lib):
    for code, name in enumerate(["GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_ALIGNMENT",
                                 "GEMM_ERR_UNSUPPORTED_DEVICE", "GEMM_ERR_CUDA",
                                 "GEMM_ERR_TIMEOUT", "GEMM_ERR_OOM"]):
        assert g.status_string(code) == name
    assert g.status_string(99) == "GEMM_ERR_UNKNOWN"


def test_variant_table(lib):
    from conftest import VARIANTS
    names = g.variant_names()
    assert names == VARIANTS
    assert lib.gemm_variant_name(len(names)) is None
    assert lib.gemm_variant_name(-1) is None


def test_null_plan_is_rejected_without_touching_cuda(lib):
    assert lib.gemm_run(None, None, None, None, 8, 8, 8, 0, None) == 1
    assert lib.gemm_run_host(None, None, None, None, 8, 8, 8, 0, None) == 1
    assert lib.gemm_plan_check_error(None) == 1
    assert lib.gemm_plan_set_watchdog(None, 0, -1) == 1
    assert lib.gemm_plan_destroy(None) == 0
    assert lib.gemm_plan_launch_count(None) == 0
    assert lib.gemm_plan_create(None, 0) == 1


def test_version(lib):
    assert re.match(r"\d+\.\d+\.\d+", lib.gemm_version().decode())


def test_host_buffers_are_taken_as_they_are():
    """gemm_run_host's binding passes the caller's own buffers: fp16,
    C-contiguous numpy arrays or CPU tensors.  Anything it would have to
    convert (a list, another dtype, a strided view) is refused, as is a
    read-only output, so no address handed to the library can dangle."""
    import numpy as np
    import torch
    a = np.zeros((4, 8), np.float16)
    assert g._host_ptr(a) == a.ctypes.data
    t = torch.zeros(4, 8, dtype=torch.float16)
    assert g._host_ptr(t) == t.data_ptr()
    with pytest.raises(TypeError):
        g._host_ptr([[0.0] * 8] * 4)
    with pytest.raises(ValueError):
        g._host_ptr(np.zeros((4, 8), np.float32))
    with pytest.raises(ValueError):
        g._host_ptr(np.zeros((8, 8), np.float16)[:, ::2])
    with pytest.raises(ValueError):
        g._host_ptr(torch.zeros(4, 8))
    with pytest.raises(ValueError):
        g._host_ptr(torch.zeros(8, 4, dtype=torch.float16).t())
    ro = np.zeros((4, 8), np.float16)
    ro.flags.writeable = False
    assert g._host_ptr(ro) == ro.ctypes.data
    with pytest.raises(ValueError):
        g._host_ptr(ro, writable=True)
