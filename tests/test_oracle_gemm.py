"""Pins of the oracle's dequantized fp64 GEMM (TN form, C = alpha A B^T + bias).

Checked against numpy's float64 matmul (a library routine), and the sampled
variant against the full product.  Also pins that the Hadamard transform
cancels inside the wgrad contraction when both operands share the sign vector
("Add an NVFP4 quantization converter", section "What changed").
"""
import numpy as np
import torch

import oracle
from mxfp8_block_scaled_bf16_gb300.inputs import rht_sign_vector


def _rand_bf16(M, K, seed=0, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, K, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_gemm_matches_numpy():
    rng = np.random.default_rng(0)
    A = rng.standard_normal((37, 53))
    B = rng.standard_normal((29, 53))
    bias = rng.standard_normal(29)
    got = oracle.gemm_tn_f64(A, B, alpha=0.75, bias=bias)
    np.testing.assert_allclose(got, 0.75 * A @ B.T + bias, rtol=1e-12, atol=1e-12)


def test_nvfp4_sampled_matches_full():
    a = _rand_bf16(64, 128, seed=1)
    b = _rand_bf16(48, 128, seed=2, std=0.02)
    ac, asc, Aa = oracle.nvfp4_quantize_rows(a)
    bc, bsc, Ab = oracle.nvfp4_quantize_rows(b)
    ga, gb = oracle.nvfp4_g(Aa), oracle.nvfp4_g(Ab)
    full = oracle.gemm_tn_f64(oracle.nvfp4_dequant(ac, asc, ga), oracle.nvfp4_dequant(bc, bsc, gb))
    rows = np.array([0, 5, 63, 17]); cols = np.array([0, 47, 3, 20])
    samp = oracle.gemm_tn_sampled(1, ac, asc, ga, bc, bsc, gb, 128, rows, cols)
    np.testing.assert_allclose(samp, full[rows, cols], rtol=1e-13, atol=1e-13)


def test_mxfp8_sampled_matches_full():
    a = _rand_bf16(64, 128, seed=3)
    b = _rand_bf16(32, 128, seed=4)
    ac, asc = oracle.mxfp8_quantize_rows(a)
    bc, bsc = oracle.mxfp8_quantize_rows(b)
    full = oracle.gemm_tn_f64(oracle.mxfp8_dequant(ac, asc), oracle.mxfp8_dequant(bc, bsc))
    rows = np.arange(0, 64, 7); cols = np.arange(0, 32, 4)[: rows.size].repeat(1)
    cols = np.resize(cols, rows.size)
    samp = oracle.gemm_tn_sampled(2, ac, asc, 1.0, bc, bsc, 1.0, 128, rows, cols)
    np.testing.assert_allclose(samp, full[rows, cols], rtol=1e-13, atol=1e-13)


def test_quantized_gemm_approximates_bf16_product():
    a = _rand_bf16(128, 256, seed=5)
    b = _rand_bf16(128, 256, seed=6)
    ac, asc, Aa = oracle.nvfp4_quantize_rows(a)
    bc, bsc, Ab = oracle.nvfp4_quantize_rows(b)
    q = oracle.gemm_tn_f64(oracle.nvfp4_dequant(ac, asc, oracle.nvfp4_g(Aa)),
                           oracle.nvfp4_dequant(bc, bsc, oracle.nvfp4_g(Ab)))
    ref = _f32(a).astype(np.float64) @ _f32(b).astype(np.float64).T
    rel = np.linalg.norm(q - ref) / np.linalg.norm(ref)
    assert rel < 0.2  # fp4 quantization noise, not a structural error


def test_rht_cancels_in_wgrad_contraction():
    """dW = dy^T x computed from RHT'd, quantized colwise operands approximates
    the plain product; with mismatched sign vectors it does not."""
    M, N, K = 256, 64, 64
    dy = _rand_bf16(M, N, seed=7)
    x = _rand_bf16(M, K, seed=8)
    ref = _f32(dy).astype(np.float64).T @ _f32(x).astype(np.float64)
    s = rht_sign_vector(7)

    def wgrad(s_dy, s_x):
        dc, ds, Ad = oracle.nvfp4_quantize_cols(dy, rht_sign=s_dy)
        xc, xs, Ax = oracle.nvfp4_quantize_cols(x, rht_sign=s_x)
        return oracle.gemm_tn_f64(oracle.nvfp4_dequant(dc, ds, oracle.nvfp4_g(Ad)),
                                  oracle.nvfp4_dequant(xc, xs, oracle.nvfp4_g(Ax)))

    good = np.linalg.norm(wgrad(s, s) - ref) / np.linalg.norm(ref)
    s2 = s.copy(); s2[:8] = -s2[:8]
    bad = np.linalg.norm(wgrad(s, s2) - ref) / np.linalg.norm(ref)
    assert good < 0.2 and bad > 0.5


def test_blas_gemm_equals_loop_gemm():
    """The numpy-matmul form computes the same fp64 product as the loop form
    (only the summation order differs)."""
    rng = np.random.default_rng(7)
    A = rng.standard_normal((70, 96))
    B = rng.standard_normal((33, 96))
    np.testing.assert_allclose(oracle.gemm_tn_f64_blas(A, B), oracle.gemm_tn_f64(A, B), rtol=1e-12, atol=1e-12)
