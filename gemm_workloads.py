"""Seeded synthetic inputs for the dense fp16 GEMM C = A @ B.T.

This module only draws and lays out inputs: it holds none of the GEMM's
arithmetic, and both the CPU oracle's tests and the CUDA path's tests and
benchmark take their operands from here.

Operands are fp16, K-major: A is [M, K] and B is [N, K], each row-major with
K contiguous (tilus "A Minimal Hopper Matmul", the "Data layout: K-major"
note).  Entries are drawn in float32 with numpy's PCG64 generator, scaled so
that each product A[i,k]*B[j,k] has variance 1/K and C has unit variance, and
cast to fp16 with round-to-nearest-even:

* "normal":  N(0,1) * K**-0.25
* "uniform": U(-1,1) * sqrt(3) * K**-0.25   (same unit variance)

A is drawn first and B second from one generator seeded with ``seed``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist: str                 # "normal" | "uniform"
    accs: tuple               # accumulations exercised: subset of ("f32", "f16")
    sample_rows: int = 0      # >0: parity on this many seeded rows + columns
    sample_seed: int = -1

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def describe(self) -> str:
        return f"C=A.B^T M={self.M} N={self.N} K={self.K} fp16 K-major, {self.dist} seed {self.seed}"


# The five workloads: a small one the oracle finishes in well under a second,
# the 4096^3 and 8192^3 squares, a ragged shape with no dimension a multiple of
# a tile (K a multiple of 8 so rows stay 16-byte aligned), and 16384^3 checked
# on seeded rows and columns.
WORKLOADS = {
    w.name: w for w in (
        Workload("gemm_512", 512, 512, 512, 0, "normal", ("f32",)),
        Workload("gemm_4096", 4096, 4096, 4096, 1, "normal", ("f32",), 256, 1001),
        Workload("gemm_8192", 8192, 8192, 8192, 2, "normal", ("f32", "f16"), 256, 1002),
        Workload("gemm_ragged_3000x5000x4104", 3000, 5000, 4104, 3, "uniform", ("f32",), 256, 1003),
        Workload("gemm_16384", 16384, 16384, 16384, 4, "normal", ("f32",), 256, 1004),
    )
}


def draw(M: int, N: int, K: int, seed: int, dist: str = "normal"):
    """Return (A [M,K], B [N,K]) as C-contiguous numpy float16 arrays."""
    rng = np.random.default_rng(seed)
    scale = np.float32(K ** -0.25) if K > 0 else np.float32(1.0)

    def one(rows):
        if dist == "normal":
            x = rng.standard_normal((rows, K), dtype=np.float32)
        elif dist == "uniform":
            x = rng.random((rows, K), dtype=np.float32)
            x *= np.float32(2.0)
            x -= np.float32(1.0)
            x *= np.float32(math.sqrt(3.0))
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        x *= scale
        return x.astype(np.float16)

    a = one(M)
    b = one(N)
    return a, b


def inputs_for(w: Workload):
    return draw(w.M, w.N, w.K, w.seed, w.dist)


def sample_indices(n: int, count: int, seed: int) -> np.ndarray:
    """``count`` distinct sorted indices in [0, n), from their own seed.
    The last index (n-1) is always included so the ragged edge tile is hit."""
    rng = np.random.default_rng(seed)
    count = min(count, n)
    idx = rng.choice(n, size=count, replace=False)
    if n - 1 not in idx:
        idx[-1] = n - 1
    return np.unique(idx).astype(np.int64)


# --- structured inputs with closed-form products (exact in fp16 and fp32) ---

def ones(M: int, N: int, K: int):
    return np.ones((M, K), np.float16), np.ones((N, K), np.float16)


def identity(n: int) -> np.ndarray:
    return np.eye(n, dtype=np.float16)


def permutation(n: int, k: int, seed: int):
    """B [n, k] with B[j, perm[j]] = 1: row j of B selects column perm[j].
    Needs n <= k; returns (B, perm)."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(k)[:n]
    b = np.zeros((n, k), np.float16)
    b[np.arange(n), perm] = 1
    return b, perm


def rank1(M: int, N: int, K: int, seed: int):
    """A[i,k] = u_i * w_k and B[j,k] = v_j * z_k with small integers, so every
    entry and every partial sum stays an exactly representable integer."""
    rng = np.random.default_rng(seed)
    u = rng.integers(-2, 3, M)
    v = rng.integers(-2, 3, N)
    w = rng.integers(-1, 2, K)
    z = rng.integers(-1, 2, K)
    a = (u[:, None] * w[None, :]).astype(np.float16)
    b = (v[:, None] * z[None, :]).astype(np.float16)
    return a, b, (u, v, w, z)
