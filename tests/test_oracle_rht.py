"""Pins of the oracle's 16-point random Hadamard transform.

"Add an NVFP4 quantization converter", section "What changed": the
Hadamard basis is shared by both GEMM operands through one sign vector, and
the transform only cancels when both operands use the same vector.  Checked
against scipy's Sylvester Hadamard matrix, H H^T = 16 I, orthogonality of T,
and the failure of the identity with different sign vectors.
"""
import numpy as np
import scipy.linalg

import oracle
from mxfp8_block_scaled_bf16_gb300.inputs import rht_sign_vector


def test_butterfly_gives_sylvester_rows():
    H = scipy.linalg.hadamard(16)
    ones = np.ones(16, dtype=np.int8)
    rows = np.stack([oracle.rht16(np.eye(16)[i], ones) for i in range(16)]) * 4.0
    assert np.array_equal(rows, H.T)  # T(e_i) * 4 = column i of H (H is symmetric)
    assert np.array_equal(rows @ rows.T, 16 * np.eye(16))


def test_matches_matrix_form_with_signs():
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = rht_sign_vector(7)
    rng = np.random.default_rng(1)
    # values on a coarse lattice so the fp32 butterfly is exact
    u = rng.integers(-64, 64, 16).astype(np.float32) / 8
    got = oracle.rht16(u, s)
    want = 0.25 * H @ (s.astype(np.float64) * u.astype(np.float64))
    assert np.array_equal(got.astype(np.float64), want)


def test_orthogonal_when_signs_shared():
    s = rht_sign_vector(7)
    rng = np.random.default_rng(3)
    for _ in range(50):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        ta = oracle.rht16(a, s).astype(np.float64)
        tb = oracle.rht16(b, s).astype(np.float64)
        assert abs(ta @ tb - a.astype(np.float64) @ b.astype(np.float64)) < 1e-5 * (1 + np.abs(a) @ np.abs(b))


def test_does_not_cancel_with_different_signs():
    s1 = rht_sign_vector(7)
    s2 = s1.copy()
    s2[3] = -s2[3]
    rng = np.random.default_rng(4)
    errs = []
    for _ in range(50):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        ta = oracle.rht16(a, s1).astype(np.float64)
        tb = oracle.rht16(b, s2).astype(np.float64)
        errs.append(abs(ta @ tb - a.astype(np.float64) @ b.astype(np.float64)))
    assert max(errs) > 0.1


def test_sign_vector_recipe():
    s = rht_sign_vector(7)
    assert s.shape == (16,) and set(np.unique(s)) <= {-1, 1}
    assert np.array_equal(s, rht_sign_vector(7))
