"""Pins for the oracle's block Hadamard rotation (CPU only)."""
import numpy as np
import pytest
import scipy.linalg

from oracle import hadamard
from oracle.formats import bf16_round


@pytest.mark.parametrize("b", [16, 64, 256])
def test_sylvester_is_orthogonal_and_matches_scipy(b):
    h = hadamard.sylvester(b)
    np.testing.assert_array_equal(h, scipy.linalg.hadamard(b).astype(np.float64))
    np.testing.assert_array_equal(h @ h.T, b * np.eye(b))


@pytest.mark.parametrize("b", [16, 64, 256])
def test_fwht_of_unit_vectors_is_normalised_hadamard(b):
    eye = np.eye(b, dtype=np.float32)
    got = hadamard.fwht_blocks(eye, b).astype(np.float64)
    np.testing.assert_array_equal(got, scipy.linalg.hadamard(b) / np.sqrt(b))


@pytest.mark.parametrize("b", [16, 64, 256])
def test_fwht_is_an_involution_on_small_integers(b):
    rng = np.random.default_rng(b)
    x = rng.integers(-8, 9, size=(5, 4 * b)).astype(np.float32)
    y = hadamard.fwht_blocks(hadamard.fwht_blocks(x, b), b)
    np.testing.assert_array_equal(y, x)


@pytest.mark.parametrize("b", [16, 64, 256])
def test_fwht_matches_dense_product(b):
    rng = np.random.default_rng(1 + b)
    x = bf16_round(rng.standard_normal((8, 2 * b)).astype(np.float32))
    got = hadamard.fwht_blocks(x, b).astype(np.float64)
    ref = hadamard.rotate_dense(x, b)
    lg = int(np.log2(b))
    tol = lg * 2.0 ** -24 * np.sqrt(b) * np.abs(x).max()
    assert np.max(np.abs(got - ref)) <= tol


@pytest.mark.parametrize("b", [16, 64, 256])
def test_rotation_preserves_inner_products(b):
    rng = np.random.default_rng(2 + b)
    x = rng.standard_normal((6, 3 * b))
    w = rng.standard_normal((7, 3 * b))
    xr, wr = hadamard.rotate_dense(x, b), hadamard.rotate_dense(w, b)
    np.testing.assert_allclose(xr @ wr.T, x @ w.T, rtol=1e-12, atol=1e-12 * np.abs(x @ w.T).max())


@pytest.mark.parametrize("b", [16, 64, 256])
def test_one_hot_outlier_is_spread(b):
    a = np.float32(96.0)
    x = np.zeros((1, b), np.float32)
    x[0, 3] = a
    y = hadamard.fwht_blocks(x, b)
    np.testing.assert_array_equal(np.abs(y), np.full((1, b), a / np.sqrt(b), np.float32))
    # max/mean ratio falls from b to 1
    ratio = lambda v: np.abs(v).max() / np.abs(v).mean()
    assert ratio(x) == b and ratio(y) == 1


def test_fwht_blocks_are_independent():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    y = hadamard.fwht_blocks(x, 16)
    for j in range(4):
        np.testing.assert_array_equal(y[:, 16 * j:16 * j + 16], hadamard.fwht_blocks(x[:, 16 * j:16 * j + 16], 16))
