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


# ------------------------------------------------------------------ H16 ----
# Fixed-sign H16 (Sec. 2.5: the NVFP4 Wgrad transform, the 16 signs applied
# once) and plain H16 (Sec. 3.3: the operand-wise hybrid's Wgrad transform,
# D = I), pinned against an independent Sylvester matrix.

def _kron_h16():
    h2 = np.array([[1, 1], [1, -1]], dtype=np.int64)
    h = np.array([[1]], dtype=np.int64)
    for _ in range(4):
        h = np.kron(h2, h)
    return h


def test_h16_butterfly_equals_matrix_product():
    # integer inputs make the binary32 butterflies exact; the final 0.25 is exact
    H = _kron_h16()
    rng = np.random.default_rng(11)
    for signs in (np.ones(16, np.int8), hadamard_signs(5)):
        d = signs.astype(np.int64)
        for _ in range(200):
            x = rng.integers(-1000, 1000, 16)
            want = (H @ (d * x)).astype(np.float64) * 0.25
            got = oracle.hadamard16_f32(x.astype(np.float32), signs).astype(np.float64)
            assert np.array_equal(got, want)


def test_plain_h16_rows_are_the_scaled_sylvester_rows():
    H = _kron_h16()
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        got = oracle.hadamard16_f32(e, np.ones(16, np.int8))
        assert np.array_equal(got.astype(np.float64) * 4.0, H[:, j].astype(np.float64))


def test_h16_is_orthonormal_and_preserves_dot():
    d = hadamard_signs(6).astype(np.float64)
    R = np.stack([oracle.hadamard16_f32(np.eye(16, dtype=np.float32)[j], hadamard_signs(6)) for j in range(16)],
                 axis=1).astype(np.float64)
    assert np.array_equal(R, _kron_h16().astype(np.float64) @ np.diag(d) / 4.0)
    assert np.array_equal(R.T @ R, np.eye(16))
    rng = np.random.default_rng(12)
    a, b = rng.standard_normal(16), rng.standard_normal(16)
    assert abs((R @ a) @ (R @ b) - a @ b) <= 1e-12 * np.abs(a * b).sum()


def test_h16_column_view_quantizes_the_transformed_blocks():
    # the column view with H16 is the untransformed quantizer applied to the
    # tensor whose every aligned 16-value column block went through H16
    rng = np.random.default_rng(13)
    x = (rng.integers(-4, 4, (64, 128)) * 2.0 ** -3).astype(np.float32)   # 16-sums stay bf16-exact
    from synthetic import bf16_bits_from_f32, f32_from_bf16_bits
    xb = bf16_bits_from_f32(x)
    xf = f32_from_bf16_bits(xb)
    signs = hadamard_signs(7)
    t = xf.T.copy()
    for r in range(t.shape[0]):
        for b0 in range(0, t.shape[1], 16):
            t[r, b0:b0 + 16] = oracle.hadamard16_f32(t[r, b0:b0 + 16], signs)
    tb = bf16_bits_from_f32(t)
    assert np.array_equal(f32_from_bf16_bits(tb), t)  # the transformed values are bf16-exact here
    for route in ("mx", "nv_global", "nv_local"):
        got = oracle.quantize(xb, route, "col", hadamard16=True, signs=signs)
        want = oracle.quantize(np.ascontiguousarray(tb.T), route, "col")
        assert np.array_equal(got["codes"], want["codes"]), route
        assert np.array_equal(got["scales"], want["scales"]), route
        if want["senc"] is not None:
            assert np.array_equal(got["senc"], want["senc"]), route
