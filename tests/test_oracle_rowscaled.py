"""Pins of the oracle's row-scaled NVFP4 ("Hybrid quantization", Description:
the grouped GEMM recipe's input quantizer NVFP4Quantizer(row_scaled_nvfp4=
True)), read as an FP32 outer scale per row instead of per tensor."""
import numpy as np
import torch

import oracle
from mxfp8_block_scaled_bf16_gb300 import inputs


def _x(M, K, seed, std=1.0):
    return inputs.normal_bf16((M, K), std, torch.Generator().manual_seed(seed))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_each_row_is_a_per_tensor_quantization_of_that_row():
    """Row-scaled quantization of a matrix = the rows quantized one by one as
    1-row tensors with the per-tensor recipe (the outer scale is the row's)."""
    x = inputs.student_t3_outliers(24, 96)
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(x)
    xb = _bits(x)
    for r in range(24):
        cr, sr_, Ar = oracle.nvfp4_quantize_rows(xb[r:r + 1])
        assert a[r] == np.float32(Ar)
        assert np.array_equal(c[r:r + 1], cr) and np.array_equal(s[r:r + 1], sr_)


def test_equals_the_per_tensor_form_when_rows_share_the_amax():
    x = _x(32, 64, 1).float().clamp(-3, 3)
    x[:, 7] = 5.0  # every row's amax is 5
    x = x.to(torch.bfloat16)
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(x)
    ct, st, At = oracle.nvfp4_quantize_rows(x)
    assert At == 5.0 and np.all(a == 5.0)
    assert np.array_equal(c, ct) and np.array_equal(s, st)


def test_row_scaled_round_trip_is_exact_on_representable_rows():
    """Row r holds E2M1 grid values times powers of two per block and one
    2688 * 2^k_r: every row dequantizes back exactly with its own scale."""
    rng = np.random.default_rng(3)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    x = np.zeros((8, 64))
    for r in range(8):
        k = int(rng.integers(-3, 4))
        for j in range(1, 4):
            sc = 2.0 ** (k + int(rng.integers(-2, 1)))
            blk = rng.choice(grid, 16) * rng.choice([-1, 1], 16)
            blk[rng.integers(16)] = 6.0
            x[r, 16 * j:16 * j + 16] = blk * sc
        x[r, 0] = 2688.0 * 2.0 ** k
    xt = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(xt)
    assert np.array_equal(oracle.nvfp4_dequant_rowscaled(c, s, a), x)


def test_zero_row_quantizes_to_zero():
    x = _x(4, 32, 2)
    x[2] = 0
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(x)
    assert a[2] == 0 and not c[2].any() and not s[2].any()
    assert not oracle.nvfp4_dequant_rowscaled(c, s, a)[2].any()


def test_sampled_gemm_matches_the_full_product():
    a = _x(48, 128, 4)
    b = _x(40, 128, 5, std=0.02)
    ac, asc, aa = oracle.nvfp4_quantize_rows_rowscaled(a)
    bc, bsc, Ab = oracle.nvfp4_quantize_rows(b)
    full = oracle.nvfp4_dequant_rowscaled(ac, asc, aa) @ oracle.nvfp4_dequant(bc, bsc, oracle.nvfp4_g(Ab)).T
    rows = np.array([0, 47, 13, 5]); cols = np.array([0, 39, 21, 7])
    got = oracle.gemm_tn_sampled_rowscaled(ac, asc, aa, bc, bsc, Ab, 128, rows, cols)
    np.testing.assert_allclose(got, full[rows, cols], rtol=1e-13, atol=1e-13)
