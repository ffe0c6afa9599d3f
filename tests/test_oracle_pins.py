"""Pins for the CPU oracle: every check here is a fact fixed independently of
the oracle's own code (numpy's binary16 conversions, exact rational sums,
closed forms, a hand-worked fixture), chosen so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails at least one.

The GEMM being pinned is C = A x B^T with A [M,K], B [N,K] K-contiguous
(tilus "A Minimal Hopper Matmul", section "Block Tiling" and the K-major note).
"""
from fractions import Fraction

import numpy as np
import pytest

import gemm_workloads as wl
import oracle
from conftest import read_golden


# ---------------------------------------------------------------- binary16 --

def test_decode_matches_numpy_on_all_65536_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_encode_roundtrips_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    assert np.array_equal(oracle.encode_f16(vals[finite]), bits[finite])


def test_encode_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(7)
    # random magnitudes over the whole fp16 range including subnormals and overflow
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
        rng.uniform(65504, 65600, 2000),
        rng.uniform(0, 2 ** -14, 2000),
    ])
    # exact ties: midpoints between neighbouring fp16 values
    lo = np.arange(0, 0x7bff, 37, dtype=np.uint16)
    mids = (lo.view(np.float16).astype(np.float64) + (lo + 1).view(np.float16).astype(np.float64)) / 2
    x = np.concatenate([x, mids, -mids, [65519.999, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26, 0.0, -0.0]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode_f16(x), ref)


# --------------------------------------------------------------- the GEMM --

def test_bt_convention_hand_worked_fixture():
    mats, _ = read_golden("bt_convention_2x3x4.txt")
    a = np.array(mats["A"], np.float16)
    b = np.array(mats["B"], np.float16)
    c = oracle.gemm_f64(a, b)
    assert c.shape == (2, 4)
    assert np.array_equal(c, np.array(mats["C"]))


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_exact_rationals_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    M, N, K = (int(v) for v in rng.integers(1, 8, 3))
    a = rng.standard_normal((M, K)).astype(np.float16)
    b = rng.standard_normal((N, K)).astype(np.float16)
    c = oracle.gemm_f64(a, b)
    fa = [[Fraction(float(v)) for v in row] for row in a.astype(np.float64)]
    fb = [[Fraction(float(v)) for v in row] for row in b.astype(np.float64)]
    for i in range(M):
        for j in range(N):
            exact = sum((fa[i][k] * fb[j][k] for k in range(K)), Fraction(0))
            bound = K * 2.0 ** -53 * sum(abs(float(fa[i][k] * fb[j][k])) for k in range(K))
            assert abs(Fraction(c[i, j]) - exact) <= Fraction(bound), (i, j)


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (17, 9, 64), (65, 70, 130), (128, 1, 33)])
def test_matches_numpy_float64_matmul(shape):
    M, N, K = shape
    a, b = wl.draw(M, N, K, seed=11, dist="normal")
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    np.testing.assert_allclose(oracle.gemm_f64(a, b), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("K", [1, 8, 64, 4104, 8192])
def test_all_ones_gives_K(K):
    a, b = wl.ones(3, 5, K)
    assert np.array_equal(oracle.gemm_f64(a, b), np.full((3, 5), float(K)))


def test_identity_left_gives_B_transposed():
    K, N = 40, 23
    _, b = wl.draw(K, N, K, seed=12)
    c = oracle.gemm_f64(wl.identity(K), b)
    assert np.array_equal(c, b.astype(np.float64).T)


def test_identity_right_gives_A():
    M, K = 31, 48
    a, _ = wl.draw(M, K, K, seed=13)
    c = oracle.gemm_f64(a, wl.identity(K))
    assert np.array_equal(c, a.astype(np.float64))


def test_permutation_selects_columns_of_A():
    M, N, K = 19, 24, 40
    a, _ = wl.draw(M, N, K, seed=14)
    b, perm = wl.permutation(N, K, seed=15)
    c = oracle.gemm_f64(a, b)
    assert np.array_equal(c, a.astype(np.float64)[:, perm])


def test_rank1_closed_form():
    M, N, K = 21, 18, 300
    a, b, (u, v, w, z) = wl.rank1(M, N, K, seed=16)
    c = oracle.gemm_f64(a, b)
    s = int(np.dot(w, z))
    assert np.array_equal(c, np.outer(u, v).astype(np.float64) * s)


def test_negating_B_negates_C():
    a, b = wl.draw(9, 10, 33, seed=17)
    assert np.array_equal(oracle.gemm_f64(a, -b), -oracle.gemm_f64(a, b))


def test_zero_K_gives_zero():
    a = np.zeros((4, 0), np.float16)
    b = np.zeros((6, 0), np.float16)
    assert np.array_equal(oracle.gemm_f64(a, b), np.zeros((4, 6)))


def test_rows_and_columns_are_slices_of_the_full_product():
    a, b = wl.draw(70, 50, 96, seed=18)
    full = oracle.gemm_f64(a, b)
    rows = np.array([0, 3, 69, 41])
    cols = np.array([49, 0, 7])
    assert np.array_equal(oracle.gemm_rows_f64(a, b, rows), full[rows])
    assert np.array_equal(oracle.gemm_cols_f64(a, b, cols), full[:, cols])


def test_thread_count_does_not_change_bits():
    a, b = wl.draw(97, 61, 257, seed=19)
    one = oracle.gemm_f64(a, b, threads=1)
    many, used = oracle.gemm_f64(a, b, threads=8, return_threads=True)
    assert used >= 1
    assert np.array_equal(one, many)


def test_input_scaling_gives_unit_variance_output():
    w = wl.WORKLOADS["gemm_512"]
    a, b = wl.inputs_for(w)
    c = oracle.gemm_f64(a, b)
    assert abs(c.std() - 1.0) < 0.03
    assert abs(c.mean()) < 0.02


def test_uniform_scaling_gives_unit_variance_output():
    a, b = wl.draw(256, 256, 1032, seed=3, dist="uniform")
    c = oracle.gemm_f64(a, b)
    assert abs(c.std() - 1.0) < 0.04
