"""CPU oracle for the dense fp16 GEMM ``C = A @ B.T`` (K-major A [M,K], B [N,K]).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library in ``dense_fp16_gemm_04_gb300`` and neither imports the
other.

The arithmetic lives in ``gemm_oracle.c`` (plain C99, IEEE double, a triple
loop over the definition C[i][j] = sum_k A[i][k]*B[j][k] from the tilus
"A Minimal Hopper Matmul" page, section "Block Tiling" and its K-major
note).  This module compiles it with gcc and calls it through ctypes; numpy
arrays of fp16 bits go in, float64 arrays come out.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself: numpy's independent binary16
conversions over all 65536 patterns, exact rational brute force on tiny
shapes, and closed forms (all-ones, identity, permutation, rank-1, the
B-transposed convention on a hand-worked 2x2 case).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=gnu99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_decode_f16.restype = None
        lib.oracle_decode_f16.argtypes = [u16p, f64p, i64]
        lib.oracle_encode_f16.restype = None
        lib.oracle_encode_f16.argtypes = [f64p, u16p, i64]
        lib.oracle_gemm_f64.restype = ctypes.c_int
        lib.oracle_gemm_f64.argtypes = [u16p, u16p, i64, i64, i64, f64p, ctypes.c_int]
        for name in ("oracle_gemm_rows_f64", "oracle_gemm_cols_f64"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [u16p, u16p, i64, i64, i64, i64p, i64, f64p, ctypes.c_int]
        _lib = lib
        return lib


def _bits(x) -> np.ndarray:
    """fp16 data (numpy float16/uint16 array, or a CPU torch tensor) -> C-contiguous uint16 bits."""
    if hasattr(x, "detach"):            # torch tensor, without importing torch here
        x = x.detach().cpu().contiguous().numpy()
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"oracle wants fp16 bits, got {x.dtype}")
    return np.ascontiguousarray(x)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(a, b):
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"want A [M,K] and B [N,K], got {a.shape} and {b.shape}")
    return a.shape[0], b.shape[0], a.shape[1]


def decode_f16(bits) -> np.ndarray:
    """binary16 bit patterns -> float64, by the oracle's own decoder."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_f16(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
    return out


def encode_f16(x) -> np.ndarray:
    """float64 -> binary16 bits (round to nearest even), by the oracle's own encoder."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_encode_f16(_ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16), x.size)
    return out


def gemm_f64(a, b, threads: int = 0, return_threads: bool = False):
    """Full C = A @ B.T in double from fp16 A [M,K], B [N,K].  ``threads=0``: all cores."""
    a, b = _bits(a), _bits(b)
    M, N, K = _shapes(a, b)
    out = np.empty((M, N), dtype=np.float64)
    used = _load().oracle_gemm_f64(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                   M, N, K, _ptr(out, ctypes.c_double), int(threads))
    return (out, used) if return_threads else out


def gemm_rows_f64(a, b, rows, threads: int = 0, return_threads: bool = False):
    """Rows ``rows`` of C, shape [len(rows), N]."""
    a, b = _bits(a), _bits(b)
    M, N, K = _shapes(a, b)
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if idx.size and (idx.min() < 0 or idx.max() >= M):
        raise IndexError("row index out of range")
    out = np.empty((idx.size, N), dtype=np.float64)
    used = _load().oracle_gemm_rows_f64(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                        M, N, K, _ptr(idx, ctypes.c_int64), idx.size,
                                        _ptr(out, ctypes.c_double), int(threads))
    return (out, used) if return_threads else out


def gemm_cols_f64(a, b, cols, threads: int = 0, return_threads: bool = False):
    """Columns ``cols`` of C, shape [M, len(cols)]."""
    a, b = _bits(a), _bits(b)
    M, N, K = _shapes(a, b)
    idx = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if idx.size and (idx.min() < 0 or idx.max() >= N):
        raise IndexError("column index out of range")
    out = np.empty((idx.size, M), dtype=np.float64)
    used = _load().oracle_gemm_cols_f64(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                        M, N, K, _ptr(idx, ctypes.c_int64), idx.size,
                                        _ptr(out, ctypes.c_double), int(threads))
    out = out.T.copy()
    return (out, used) if return_threads else out


__all__ = ["build", "decode_f16", "encode_f16", "gemm_f64", "gemm_rows_f64", "gemm_cols_f64"]
