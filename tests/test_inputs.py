"""The seeded input generator: SplitMix64 draws and the value recipes built on them."""

import numpy as np

from dense_fp32_gemm_sgemm_gb300.inputs import (make_inputs, make_permutation,
                                               sample_indices, splitmix64)


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 from state 0, as published with the generator
    d = splitmix64(0, 0, 3)
    assert [int(x) for x in d] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                   0x06C45D188009454F]


def test_counter_based_offsets():
    full = splitmix64(7, 0, 100)
    assert np.array_equal(splitmix64(7, 40, 60), full[40:])


def test_uniform_values_exact_and_in_range():
    A, B = make_inputs(64, 128, 32, 0, "uniform")
    for x in (A, B):
        assert x.dtype == np.float32
        assert x.min() >= -1.0 and x.max() < 1.0
        scaled = x.astype(np.float64) * 2.0 ** 23
        assert np.array_equal(scaled, np.round(scaled))
    assert abs(float(A.mean())) < 0.05


def test_uniform01_values_exact_same_sign_and_from_the_same_draws():
    A, B = make_inputs(64, 128, 32, 5, "uniform01")
    for x in (A, B):
        assert x.dtype == np.float32
        assert x.min() >= 0.0 and x.max() < 1.0
        scaled = x.astype(np.float64) * 2.0 ** 24
        assert np.array_equal(scaled, np.round(scaled))
    assert abs(float(A.mean()) - 0.5) < 0.05
    # the same 24-bit draws as "uniform" on [-1, 1): u01 = (u + 1) / 2, exactly
    U, _ = make_inputs(64, 128, 32, 5, "uniform")
    assert np.array_equal((U.astype(np.float64) + 1.0) / 2.0, A.astype(np.float64))
    d = splitmix64(5, 0, 4)
    assert [float(A.ravel()[i]) for i in range(4)] == [int(x >> np.uint64(40)) * 2.0 ** -24
                                                       for x in d]


def test_integer_ranges_inclusive():
    A, B = make_inputs(200, 100, 50, 1, "int8")
    vals = np.unique(np.concatenate([A.ravel(), B.ravel()]))
    assert np.array_equal(vals, np.arange(-8, 9, dtype=np.float32))
    A4, _ = make_inputs(100, 100, 1, 0, "int4")
    assert np.array_equal(np.unique(A4), np.arange(-4, 5, dtype=np.float32))


def test_normal_moments():
    A, _ = make_inputs(256, 256, 1, 3, "normal")
    assert abs(float(A.mean())) < 0.02
    assert abs(float(A.std()) - 1.0) < 0.02


def test_a_independent_of_k_and_deterministic():
    A1, B1 = make_inputs(5, 7, 3, 11)
    A2, B2 = make_inputs(5, 7, 9, 11)
    assert np.array_equal(A1, A2)
    A3, B3 = make_inputs(5, 7, 3, 11)
    assert np.array_equal(B1, B3)


def test_permutation_and_samples():
    p = make_permutation(100, 3)
    assert np.array_equal(np.sort(p), np.arange(100))
    r, c = sample_indices(50, 60, 20, 1)
    assert r.shape == (24,) and c.shape == (24,)
    assert r.min() >= 0 and r.max() < 50 and c.min() >= 0 and c.max() < 60
    assert (r[:4] == [0, 0, 49, 49]).all() and (c[:4] == [0, 59, 0, 59]).all()
