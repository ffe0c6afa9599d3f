"""GB300-native dense fp16 GEMM, C = A @ B.T with K-major operands.

A thin ctypes binding over the C ABI in ``include/gemm.h``; every step of the
product runs in the sm_103a kernels of ``libgb300gemm.so`` (built in-tree from
``csrc/`` by :func:`build`).  There is no fallback: if the library is missing
or the device is not an sm_103 part, calls raise.

    >>> import torch, dense_fp16_gemm_04_gb300 as g
    >>> a = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)
    >>> b = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)
    >>> c = g.gemm(a, b)              # fp32 accumulate -> fp16
    >>> c16 = g.gemm(a, b, acc="f16")  # native fp16 accumulate

The operation (tilus "A Minimal Hopper Matmul", "Block Tiling"): A is
[M, K], B is [N, K], both row-major with K contiguous; C[i, j] =
sum_k A[i, k] * B[j, k].
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "build", "load", "Plan", "GemmError", "gemm", "gemm_host", "default_plan",
    "ACC_F32", "ACC_F16", "K_CONTIGUOUS", "MN_CONTIGUOUS", "status_string", "variant_names", "variant_info",
    "LIB_PATH",
]

LIB_PATH = _build.LIB_PATH
ACC_F32 = 0
ACC_F16 = 1
K_CONTIGUOUS = 0    # A stored [M, K], B stored [N, K]
MN_CONTIGUOUS = 1   # A stored [K, M], B stored [K, N]
_ACC = {"f32": ACC_F32, "fp32": ACC_F32, "float32": ACC_F32, ACC_F32: ACC_F32,
        "f16": ACC_F16, "fp16": ACC_F16, "float16": ACC_F16, ACC_F16: ACC_F16}

_STATUS = {
    0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_ALIGNMENT",
    3: "GEMM_ERR_UNSUPPORTED_DEVICE", 4: "GEMM_ERR_CUDA", 5: "GEMM_ERR_TIMEOUT",
    6: "GEMM_ERR_OOM",
}

_lib = None
_lib_lock = threading.Lock()


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        name = _STATUS.get(self.status, f"status {self.status}")
        super().__init__(f"{where}: {name}" if where else name)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libgb300gemm.so`` for sm_103a if its sources changed."""
    return _build.build(force=force, verbose=verbose)


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with dense_fp16_gemm_04_gb300.build() "
                "(nvcc, sm_103a); there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        st = ctypes.c_int
        sig = {
            "gemm_plan_create": (st, [ctypes.POINTER(vp), ctypes.c_int]),
            "gemm_plan_destroy": (st, [vp]),
            "gemm_run": (st, [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]),
            "gemm_run_host": (st, [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]),
            "gemm_run_ex": (st, [vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, i64, i64, i64,
                                 ctypes.c_int, vp]),
            "gemm_plan_check_error": (st, [vp]),
            "gemm_plan_last_error_detail": (st, [vp, ctypes.POINTER(ctypes.c_uint32)]),
            "gemm_plan_set_watchdog": (st, [vp, u64, i32]),
            "gemm_plan_set_variant": (st, [vp, i32]),
            "gemm_plan_set_schedule": (st, [vp, i32]),
            "gemm_plan_set_pdl": (st, [vp, i32]),
            "gemm_plan_set_tile_order": (st, [vp, i32]),
            "gemm_plan_describe": (i32, [vp, i64, i64, i64, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int64)]),
            "gemm_variant_count": (i32, []),
            "gemm_variant_name": (ctypes.c_char_p, [i32]),
            "gemm_variant_info": (i32, [i32, ctypes.POINTER(i32)]),
            "gemm_plan_resident_units": (st, [vp, ctypes.POINTER(i32)]),
            "gemm_plan_pick_variant": (i32, [vp, i64, i64, i64, ctypes.c_int,
                                             ctypes.POINTER(i32)]),
            "gemm_plan_launch_count": (u64, [vp]),
            "gemm_plan_kernel_clock": (st, [vp, ctypes.POINTER(u64)]),
            "gemm_plan_set_clock_record": (st, [vp, i32]),
            "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "gemm_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def variant_names():
    lib = load()
    return [lib.gemm_variant_name(i).decode() for i in range(lib.gemm_variant_count())]


def variant_info(variant) -> dict:
    """CTAs per unit, the unit's tile of C (rows x columns) and whether the
    MMA roles are swapped, for a variant given by name or index."""
    if isinstance(variant, str):
        variant = variant_names().index(variant)
    out = (ctypes.c_int32 * 4)()
    if load().gemm_variant_info(int(variant), out) != 0:
        raise ValueError(f"unknown variant {variant!r}")
    return {"ctas": out[0], "tile_m": out[1], "tile_n": out[2], "swap": bool(out[3])}


def _check(status: int, where: str):
    if status != 0:
        raise GemmError(status, where)


def _acc(acc) -> int:
    try:
        return _ACC[acc]
    except KeyError:
        raise ValueError(f"acc must be 'f32' or 'f16', got {acc!r}") from None


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a ``gemm_plan_t`` bound to one CUDA device."""

    def __init__(self, device: int = 0):
        self._lib = load()
        self._h = ctypes.c_void_p()
        _check(self._lib.gemm_plan_create(ctypes.byref(self._h), int(device)), "gemm_plan_create")
        self.device = int(device)

    @property
    def handle(self) -> int:
        return self._h.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.gemm_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- raw pointer interface (the C ABI, one to one) ------------------------
    def run_ptr(self, a_ptr: int, b_ptr: int, c_ptr: int, M: int, N: int, K: int,
                acc="f32", stream: int = 0) -> None:
        _check(self._lib.gemm_run(self._h, a_ptr, b_ptr, c_ptr, M, N, K, _acc(acc), stream),
               "gemm_run")

    def run_host_ptr(self, a_ptr: int, b_ptr: int, c_ptr: int, M: int, N: int, K: int,
                     acc="f32", stream: int = 0) -> None:
        _check(self._lib.gemm_run_host(self._h, a_ptr, b_ptr, c_ptr, M, N, K, _acc(acc), stream),
               "gemm_run_host")

    def run_ex_ptr(self, a_ptr: int, layout_a: int, b_ptr: int, layout_b: int, c_ptr: int,
                   M: int, N: int, K: int, acc="f32", stream: int = 0) -> None:
        _check(self._lib.gemm_run_ex(self._h, a_ptr, int(layout_a), b_ptr, int(layout_b), c_ptr,
                                     M, N, K, _acc(acc), stream), "gemm_run_ex")

    def status_run(self, a_ptr, b_ptr, c_ptr, M, N, K, acc=0, stream=0) -> int:
        """gemm_run's raw status code (no exception)."""
        return self._lib.gemm_run(self._h, a_ptr, b_ptr, c_ptr, M, N, K, int(acc), stream)

    # -- torch tensor interface ------------------------------------------------
    def run(self, a, b, c, acc="f32", stream=None) -> None:
        """C = A @ B.T on CUDA tensors: fp16, A [M,K], B [N,K], C [M,N] contiguous.
        A and B may each be contiguous or the transpose of a contiguous tensor
        (A = x.t() with x [K,M]; B = w.t() with w [K,N], i.e. C = A @ w)."""
        M, N, K, la, lb = _check_tensors(a, b, c, self.device)
        sh = _stream_handle(stream)
        if la == K_CONTIGUOUS and lb == K_CONTIGUOUS:
            self.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, acc, sh)
        else:
            self.run_ex_ptr(a.data_ptr(), la, b.data_ptr(), lb, c.data_ptr(), M, N, K, acc, sh)

    def run_host(self, a, b, c, acc="f32", stream=None) -> None:
        """Same on CPU tensors/arrays (pinned for full copy speed); synchronous."""
        if len(a.shape) != 2 or len(b.shape) != 2 or len(c.shape) != 2:
            raise ValueError("want A [M,K], B [N,K], C [M,N]")
        M, K = a.shape
        N = b.shape[0]
        if tuple(b.shape) != (N, K) or tuple(c.shape) != (M, N):
            raise ValueError("want A [M,K], B [N,K], C [M,N]")
        self.run_host_ptr(_host_ptr(a), _host_ptr(b), _host_ptr(c, writable=True), M, N, K, acc,
                          _stream_handle(stream))

    def check_error(self) -> None:
        """Synchronize; raise GemmError if a kernel's watchdog fired."""
        _check(self._lib.gemm_plan_check_error(self._h), "gemm_plan_check_error")

    def check_error_status(self) -> int:
        return self._lib.gemm_plan_check_error(self._h)

    def last_error_detail(self):
        d = (ctypes.c_uint32 * 4)()
        _check(self._lib.gemm_plan_last_error_detail(self._h, d), "gemm_plan_last_error_detail")
        return list(d)

    def set_watchdog(self, timeout_ns: int = 0, skip_k_block: int = -1) -> None:
        _check(self._lib.gemm_plan_set_watchdog(self._h, int(timeout_ns), int(skip_k_block)),
               "gemm_plan_set_watchdog")

    def set_variant(self, variant) -> None:
        if isinstance(variant, str):
            variant = variant_names().index(variant)
        _check(self._lib.gemm_plan_set_variant(self._h, int(variant)), "gemm_plan_set_variant")

    def set_schedule(self, mode) -> None:
        """'auto' (0), 'whole' tiles only (1) or 'streamk' whenever possible (2)."""
        mode = {"auto": 0, "whole": 1, "streamk": 2}.get(mode, mode)
        _check(self._lib.gemm_plan_set_schedule(self._h, int(mode)), "gemm_plan_set_schedule")

    def set_tile_order(self, mode) -> None:
        """'auto' (0), 'static' round robin (1) or 'dynamic' whenever possible (2)."""
        mode = {"auto": 0, "static": 1, "dynamic": 2}.get(mode, mode)
        _check(self._lib.gemm_plan_set_tile_order(self._h, int(mode)), "gemm_plan_set_tile_order")

    def set_pdl(self, enable: bool) -> None:
        """Programmatic dependent launch of the GEMM kernel (default on)."""
        _check(self._lib.gemm_plan_set_pdl(self._h, 1 if enable else 0), "gemm_plan_set_pdl")

    def describe(self, M, N, K, acc="f32") -> dict:
        """How gemm_run would lay out this call on the device."""
        out = (ctypes.c_int64 * 6)()
        if self._lib.gemm_plan_describe(self._h, M, N, K, _acc(acc), out) != 0:
            raise GemmError(1, "gemm_plan_describe")
        return {"variant": variant_names()[out[0]], "grid_ctas": out[1], "units": out[2],
                "dp_tiles": out[3], "sk_units": out[4], "sk_iters": out[5]}

    def pick_variant(self, M, N, K, acc="f32"):
        grid = ctypes.c_int32(0)
        v = self._lib.gemm_plan_pick_variant(self._h, M, N, K, _acc(acc), ctypes.byref(grid))
        if v < 0:
            raise GemmError(1, "gemm_plan_pick_variant")
        return variant_names()[v], grid.value

    def resident_units(self) -> dict:
        """Units of each kind that fit on the device at once."""
        out = (ctypes.c_int32 * 3)()
        _check(self._lib.gemm_plan_resident_units(self._h, out), "gemm_plan_resident_units")
        return {"ctas": out[0], "pairs": out[1], "quads": out[2]}

    def set_clock_record(self, enable: bool) -> None:
        """Kernels add to the plan's clock record (off by default)."""
        _check(self._lib.gemm_plan_set_clock_record(self._h, 1 if enable else 0),
               "gemm_plan_set_clock_record")

    def kernel_clock(self) -> dict:
        """Synchronize, then read and reset the kernels' own clock record:
        launches since the last read, CTA 0's lifetime summed in SM cycles and
        in ns, and their ratio, the mean SM clock (MHz) the kernels ran at."""
        out = (ctypes.c_uint64 * 3)()
        _check(self._lib.gemm_plan_kernel_clock(self._h, out), "gemm_plan_kernel_clock")
        launches, cycles, ns = int(out[0]), int(out[1]), int(out[2])
        return {"launches": launches, "cycles": cycles, "ns": ns,
                "mhz": cycles * 1e3 / ns if ns else None}

    @property
    def launch_count(self) -> int:
        return int(self._lib.gemm_plan_launch_count(self._h))


def _layout(t, name):
    """K_CONTIGUOUS for a contiguous [rows, K] tensor, MN_CONTIGUOUS for the
    transpose of a contiguous [K, rows] tensor."""
    if t.is_contiguous():
        return K_CONTIGUOUS
    if t.t().is_contiguous():
        return MN_CONTIGUOUS
    raise ValueError(f"{name} must be contiguous or the transpose of a contiguous tensor")


def _check_tensors(a, b, c, device=None):
    """Shapes and layouts of A, B, C; all three must live on the plan's
    device (the kernel runs there and would fault on another GPU's memory)."""
    import torch
    for name, t in (("A", a), ("B", b), ("C", c)):
        if t.dtype != torch.float16:
            raise TypeError(f"{name} must be float16, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if device is not None and t.device.index != device:
            raise ValueError(f"{name} is on cuda:{t.device.index}, the plan on cuda:{device}")
        if t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D tensor")
    if not c.is_contiguous():
        raise ValueError("C must be contiguous")
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K or tuple(c.shape) != (M, N):
        raise ValueError(f"want A [M,K], B [N,K], C [M,N]; got {tuple(a.shape)}, "
                         f"{tuple(b.shape)}, {tuple(c.shape)}")
    return M, N, K, _layout(a, "A"), _layout(b, "B")


def _host_ptr(x, writable: bool = False) -> int:
    """Address of a host buffer the library reads (or, `writable`, writes):
    a contiguous fp16 CPU tensor or numpy array.  Nothing is converted: a
    converted copy would be freed when this returns, leaving the library a
    dangling address, and an output written into a copy would be lost."""
    import numpy as np
    if hasattr(x, "data_ptr"):
        import torch
        if x.is_cuda or not x.is_contiguous() or x.dtype != torch.float16:
            raise ValueError("host tensors must be contiguous float16 CPU tensors")
        return x.data_ptr()
    if not isinstance(x, np.ndarray):
        raise TypeError("host buffers must be numpy arrays or CPU tensors, got %s"
                        % type(x).__name__)
    if x.dtype != np.float16 or not x.flags.c_contiguous:
        raise ValueError("host arrays must be C-contiguous float16")
    if writable and not x.flags.writeable:
        raise ValueError("the output array is read-only")
    return x.ctypes.data


_plans = {}
_plans_lock = threading.Lock()


def default_plan(device=None, stream=None) -> Plan:
    """One shared plan per (device, stream), created on first use: work
    launched through one plan must not overlap on the GPU."""
    import torch
    if device is None:
        device = torch.cuda.current_device()
    device = int(device)
    key = (device, _stream_handle(stream) if stream is not None
           else torch.cuda.current_stream(device).cuda_stream)
    with _plans_lock:
        p = _plans.get(key)
        if p is None:
            p = _plans[key] = Plan(device)
        return p


def gemm(a, b, acc="f32", out=None, stream=None, plan: Plan | None = None):
    """C = A @ B.T for fp16 CUDA tensors A [M,K], B [N,K]; returns C [M,N] fp16."""
    import torch
    if out is None:
        out = torch.empty((a.shape[0], b.shape[0]), dtype=torch.float16, device=a.device)
    (plan or default_plan(a.device.index, stream)).run(a, b, out, acc=acc, stream=stream)
    return out


def gemm_host(a, b, acc="f32", out=None, stream=None, plan: Plan | None = None):
    """C = A @ B.T for host (CPU) fp16 tensors; copies in, computes, copies out."""
    import torch
    if out is None:
        out = torch.empty((a.shape[0], b.shape[0]), dtype=torch.float16,
                          pin_memory=bool(getattr(a, "is_pinned", lambda: False)()))
    (plan or default_plan()).run_host(a, b, out, acc=acc, stream=stream)
    return out
