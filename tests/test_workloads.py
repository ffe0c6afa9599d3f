"""The seeded input generators: deterministic, right shapes, right scale."""
import numpy as np

import gemm_workloads as wl


def test_draw_is_deterministic_and_fp16_kmajor():
    a1, b1 = wl.draw(33, 17, 40, seed=5)
    a2, b2 = wl.draw(33, 17, 40, seed=5)
    assert a1.dtype == np.float16 and b1.dtype == np.float16
    assert a1.shape == (33, 40) and b1.shape == (17, 40)
    assert a1.flags.c_contiguous and b1.flags.c_contiguous
    assert np.array_equal(a1.view(np.uint16), a2.view(np.uint16))
    assert np.array_equal(b1.view(np.uint16), b2.view(np.uint16))
    a3, _ = wl.draw(33, 17, 40, seed=6)
    assert not np.array_equal(a1, a3)


def test_scales():
    K = 4096
    a, _ = wl.draw(64, 8, K, seed=1)
    assert abs(a.astype(np.float64).std() - K ** -0.25) < 0.01 * K ** -0.25 * 5
    u, _ = wl.draw(64, 8, K, seed=3, dist="uniform")
    bound = np.sqrt(3.0) * K ** -0.25
    assert np.abs(u.astype(np.float64)).max() <= bound * (1 + 1e-3)
    assert abs(u.astype(np.float64).std() - K ** -0.25) < 0.05 * K ** -0.25


def test_workload_table():
    names = list(wl.WORKLOADS)
    assert names[0] == "gemm_512" and len(names) == 5
    for w in wl.WORKLOADS.values():
        assert w.K % 8 == 0 and w.N % 8 == 0
    r = wl.WORKLOADS["gemm_ragged_3000x5000x4104"]
    assert (r.M % 128, r.N % 256, r.K % 64) != (0, 0, 0)
    assert wl.WORKLOADS["gemm_8192"].accs == ("f32", "f16")


def test_sample_indices():
    idx = wl.sample_indices(3000, 256, 1003)
    assert idx.dtype == np.int64 and len(idx) == 256
    assert np.all(np.diff(idx) > 0) and idx[0] >= 0 and idx[-1] == 2999
    assert np.array_equal(idx, wl.sample_indices(3000, 256, 1003))


def test_structured_inputs():
    b, perm = wl.permutation(5, 9, seed=0)
    assert (b.sum(axis=1) == 1).all() and len(set(perm.tolist())) == 5
    a, b, (u, v, w, z) = wl.rank1(4, 3, 10, seed=0)
    assert np.array_equal(a.astype(np.int64), np.outer(u, w))
