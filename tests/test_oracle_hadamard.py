"""Pins of the oracle's fixed-sign H32 (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 2.5 Eq. 10, Appendix A.1): R = H D / sqrt(32) is orthogonal,
so the paired transform preserves the unquantized Wgrad dot product."""
import numpy as np
import pytest

import oracle
from synthetic import hadamard_signs


def _kron_h32():
    h2 = np.array([[1, 1], [1, -1]], dtype=np.int64)
    h = np.array([[1]], dtype=np.int64)
    for _ in range(5):
        h = np.kron(h2, h)
    return h


def test_sylvester_h32_is_kronecker_power_and_orthogonal():
    h = oracle.sylvester_h32().astype(np.int64)
    assert np.array_equal(h, _kron_h32())
    assert set(np.unique(h)) == {-1, 1}
    assert np.array_equal(h.T @ h, 32 * np.eye(32, dtype=np.int64))


def test_signed_transform_is_orthonormal_and_preserves_dot(paper_facts):
    assert paper_facts["hadamard_half_signs"] == 16
    d16 = hadamard_signs(1)
    D = np.diag(np.tile(d16, 2).astype(np.float64))
    R = oracle.sylvester_h32().astype(np.float64) @ D / np.sqrt(32.0)
    assert np.abs(R.T @ R - np.eye(32)).max() < 1e-15
    rng = np.random.default_rng(0)
    a, b = rng.standard_normal(32), rng.standard_normal(32)
    assert abs((R @ a) @ (R @ b) - a @ b) <= 1e-12 * np.abs(a * b).sum()


def test_butterfly_equals_matrix_product():
    # integer inputs: the binary32 butterflies are exact, so the oracle's output
    # equals fl32(H D x) * fl32(1/sqrt(32)) computed from the explicit matrix
    d16 = hadamard_signs(2)
    H = oracle.sylvester_h32().astype(np.int64)
    D = np.tile(d16, 2).astype(np.int64)
    s = np.float32(oracle.inv_sqrt32_f32())
    assert s == np.float32(2.0 ** -2.5)
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = rng.integers(-1000, 1000, 32)
        exact = (H @ (D * x)).astype(np.float32)
        ref = (exact * s).astype(np.float32)
        got = oracle.hadamard32_f32(x.astype(np.float32), d16)
        assert np.array_equal(got, ref)


def test_one_hot_columns_follow_signs():
    d16 = hadamard_signs(3)
    H = oracle.sylvester_h32()
    for j in range(32):
        e = np.zeros(32, np.float32)
        e[j] = 1.0
        got = oracle.hadamard32_f32(e, d16)
        want = (H[:, j] * d16[j % 16]).astype(np.float32) * np.float32(oracle.inv_sqrt32_f32())
        assert np.array_equal(got, want)


def test_general_inputs_within_binary32_rounding():
    d16 = hadamard_signs(4)
    R = oracle.sylvester_h32().astype(np.float64) @ np.diag(np.tile(d16, 2).astype(np.float64)) / np.sqrt(32)
    rng = np.random.default_rng(2)
    for _ in range(200):
        x = (rng.standard_normal(32) * np.exp(rng.uniform(-5, 5, 32))).astype(np.float32)
        got = oracle.hadamard32_f32(x, d16).astype(np.float64)
        ref = R @ x.astype(np.float64)
        bound = 8 * 2.0 ** -24 * np.abs(x).sum()
        assert np.abs(got - ref).max() <= bound
