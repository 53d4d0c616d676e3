"""Pins of the oracle's 16-point random Hadamard transform."""
import numpy as np
import pytest
import scipy.linalg

import oracle

MASK = oracle.DEFAULT_SIGN_MASK


def sigma(mask):
    return np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])


def test_matches_sylvester_matrix_product():
    """y = 1/4 * H16 * diag(sigma) * d, with H16 from scipy's Sylvester
    construction; the FP32 butterflies agree with the float64 product to FP32
    rounding (and exactly on integer inputs, where every sum is exact)."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    assert np.array_equal(H, np.kron(np.kron(np.kron([[1, 1], [1, -1]], [[1, 1], [1, -1]]),
                                             [[1, 1], [1, -1]]), [[1, 1], [1, -1]]))
    rng = np.random.default_rng(0)
    for mask in (0, MASK, 0xFFFF, 0x0001):
        for _ in range(200):
            d = rng.standard_normal(16).astype(np.float32)
            y = oracle.rht16_f32(d, mask).astype(np.float64)
            ref = 0.25 * H @ (sigma(mask) * d.astype(np.float64))
            assert np.allclose(y, ref, rtol=0, atol=4 * 2.0 ** -24 * np.abs(d).sum())
        d = rng.integers(-1000, 1000, 16).astype(np.float32)
        y = oracle.rht16_f32(d, mask).astype(np.float64)
        np.testing.assert_array_equal(y, 0.25 * H @ (sigma(mask) * d.astype(np.float64)))


def test_orthonormal_inverse_and_parseval():
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(1)
    d = rng.standard_normal(16).astype(np.float32)
    y = oracle.rht16_f32(d, MASK).astype(np.float64)
    back = sigma(MASK) * (0.25 * H @ y)
    assert np.allclose(back, d, atol=1e-6)
    assert np.isclose((y ** 2).sum(), (d.astype(np.float64) ** 2).sum(), rtol=1e-6)


def test_tight_4x_case_and_single_spike():
    """d_i = a * sigma_i gives y_0 = 4a and y_i = 0 otherwise: the case where
    the post-RHT amax reaches 4x the input amax.  A single nonzero d_l gives
    |y_i| = |d_l| / 4 for every i."""
    a = 1.75
    y = oracle.rht16_f32((a * sigma(MASK)).astype(np.float32), MASK)
    assert y[0] == 4 * a and np.all(y[1:] == 0)
    for l in range(16):
        d = np.zeros(16, np.float32)
        d[l] = -3.0
        y = oracle.rht16_f32(d, MASK)
        assert np.all(np.abs(y) == 0.75)


def test_bound_holds_on_random_blocks():
    rng = np.random.default_rng(2)
    for _ in range(2000):
        d = (rng.standard_normal(16) * np.exp(rng.standard_normal(16))).astype(np.float32)
        y = oracle.rht16_f32(d, MASK)
        assert np.abs(y).max() <= 4 * np.abs(d).max()
