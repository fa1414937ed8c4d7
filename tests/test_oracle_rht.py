"""Pins for the oracle's random Hadamard transform (CPU only).

The 16-point transform must be 1/4 * H16 * diag(sigma) with H16 the
Sylvester Hadamard matrix, so that H16 H16^T = 16 I and the transform is
orthogonal ("Full-Stack FP4...", section 2.2 uses Hadamard mixing to spread
outliers before quantisation).
"""
import numpy as np

import oracle


def _sylvester(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _oracle_matrix(sigma):
    cols = []
    for j in range(16):
        e = np.zeros(16, dtype=np.float32)
        e[j] = 1.0
        cols.append(oracle.rht16(e, sigma).astype(np.float64))
    return np.stack(cols, axis=1)


def test_transform_is_quarter_sylvester_times_signs():
    for seed in (0, 1, 12345, 2 ** 63 + 5):
        sigma = oracle.rht_signs(seed)
        assert set(np.unique(sigma)) <= {-1.0, 1.0}
        h = _oracle_matrix(sigma)
        assert np.array_equal(h, 0.25 * _sylvester(16) @ np.diag(sigma.astype(np.float64)))


def test_hadamard_orthogonality():
    h = 4.0 * _oracle_matrix(np.ones(16, dtype=np.float32))
    assert np.array_equal(h @ h.T, 16.0 * np.eye(16))


def test_signs_come_from_philox_word0():
    seed = 0xDEADBEEF12345678
    w = oracle.philox4x32_10([0, 0, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])[0]
    sigma = oracle.rht_signs(seed)
    for j in range(16):
        assert sigma[j] == (-1.0 if (int(w) >> j) & 1 else 1.0)
    assert not np.array_equal(oracle.rht_signs(1), oracle.rht_signs(2))


def test_norm_preserved_and_inverse():
    rng = np.random.default_rng(0)
    sigma = oracle.rht_signs(7)
    for _ in range(200):
        x = rng.standard_normal(16).astype(np.float32)
        y = oracle.rht16(x, sigma)
        assert abs(np.linalg.norm(y.astype(np.float64)) - np.linalg.norm(x.astype(np.float64))) < 1e-5 * np.linalg.norm(x)
        # inverse of 1/4 H diag(s) is diag(s) 1/4 H (H symmetric, H H = 16 I)
        back = oracle.rht16(y, np.ones(16, dtype=np.float32)) * sigma
        assert np.allclose(back, x, atol=1e-6, rtol=1e-6)


def test_integer_vectors_are_exact():
    rng = np.random.default_rng(1)
    sigma = oracle.rht_signs(99)
    for _ in range(50):
        x = rng.integers(-64, 64, size=16).astype(np.float32)
        y = oracle.rht16(x, sigma).astype(np.float64)
        assert np.array_equal(y, 0.25 * _sylvester(16) @ (sigma.astype(np.float64) * x))


def test_shared_signs_cancel_in_inner_products():
    # (1/4 H D a) . (1/4 H D b) = a . b, which is why both wgrad operands use
    # the same sign vector.
    rng = np.random.default_rng(2)
    sigma = oracle.rht_signs(2024)
    a = rng.standard_normal(16).astype(np.float32)
    b = rng.standard_normal(16).astype(np.float32)
    lhs = float(np.dot(oracle.rht16(a, sigma).astype(np.float64), oracle.rht16(b, sigma).astype(np.float64)))
    assert abs(lhs - float(np.dot(a.astype(np.float64), b.astype(np.float64)))) < 1e-5
