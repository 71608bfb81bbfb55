"""Pins of the oracle's rowwise-dequantized source and identity direction
("Hybrid quantization", "Enable columnwise_source and hybrid recipes": with
columnwise_source="rowwise_dequantized" the columnwise operand is built from
dequantize(rowwise-quantized x); IdentityQuantizer passes the high-precision
value through; the review's test that the rowwise-dequantized source with an
identity columnwise quantizer matches the rowwise value)."""
import numpy as np
import torch

import oracle
from mxfp8_block_scaled_bf16_gb300 import inputs


def _x(M, K, seed, std=1.0):
    return inputs.normal_bf16((M, K), std, torch.Generator().manual_seed(seed))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _e2m1_table():
    return np.array([oracle.e2m1_decode(c) for c in range(16)], np.float64)


def test_nvfp4_dequant_matches_fp32_numpy_and_torch_cast():
    """Independent restatement with library arithmetic: numpy's fp32 multiply
    of the exact E2M1 x E4M3 product by g = fl(A / 2688), then torch's
    fp32 -> bf16 cast (round to nearest even)."""
    x = _x(96, 128, 1)
    c, s, A = oracle.nvfp4_quantize_rows(x)
    lo, hi = c & 15, c >> 4
    codes = np.empty((96, 128), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    e4 = np.array([oracle.e4m3_decode(v) for v in range(256)], np.float64)
    cs = (_e2m1_table()[codes] * np.repeat(e4[s], 16, axis=1)).astype(np.float32)
    g = np.float32(A) / np.float32(2688.0)
    v = cs * g  # numpy fp32 multiply, one rounding
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.nvfp4_dequant_bf16(c, s, A), want)


def test_nvfp4_dequant_equals_fp64_dequant_when_g_is_a_power_of_two():
    """With A = 2688 * 2^k the fp32 product is exact, so the bf16 value is the
    fp64 dequantized value rounded once."""
    x = _x(64, 64, 2).float()
    x[3, 5] = 2688.0 * 0.25
    x = x.to(torch.bfloat16)
    c, s, A = oracle.nvfp4_quantize_rows(x)
    assert A == 672.0
    got = oracle.nvfp4_dequant_bf16(c, s, A)
    assert np.array_equal(got, oracle.to_bf16_rne(oracle.nvfp4_dequant(c, s, oracle.nvfp4_g(A))))


def test_mxfp8_dequant_is_exact_and_requantizes_to_the_same_operand():
    """E4M3 x 2^e is exact, and an MXFP8 block whose values are already
    E4M3 x 2^e quantizes to the same codes and scale again (idempotence)."""
    x = inputs.student_t3_outliers(128, 256)
    c, s = oracle.mxfp8_quantize_rows(x)
    xd = oracle.mxfp8_dequant_bf16(c, s)
    assert np.array_equal(xd, oracle.to_bf16_rne(oracle.mxfp8_dequant(c, s)))
    c2, s2 = oracle.mxfp8_quantize_rows(xd)
    assert np.array_equal(c2, c) and np.array_equal(s2, s)


def test_identity_direction_is_the_value_itself():
    x = _x(40, 48, 3)
    xb = _bits(x)
    assert np.array_equal(oracle.identity_rows(x), xb)
    cols = oracle.identity_cols(x)
    assert cols.shape == (48, 48)
    assert np.array_equal(cols[:, :40], xb.T) and not cols[:, 40:].any()


def test_rowwise_dequantized_identity_columnwise_matches_rowwise():
    """The review's double-quantization test: with the rowwise-dequantized
    source, the identity columnwise operand is the rowwise dequantized value
    (transposed into the K-major columnwise layout)."""
    x = _x(64, 96, 4)
    for fmt in (1, 2):
        xd, _ = oracle.rowwise_dequantized(x, fmt)
        assert np.array_equal(oracle.identity_cols(xd), xd.T)


def test_double_quantization_differs_from_the_original_source():
    """Quantizing the dequantized value columnwise is not the same as quantizing
    the original: the backward sees the forward's quantization error."""
    x = _x(128, 128, 5)
    xd, _ = oracle.rowwise_dequantized(x, 1)
    c_orig, _ = oracle.mxfp8_quantize_cols(x)
    c_dq, _ = oracle.mxfp8_quantize_cols(xd)
    assert not np.array_equal(c_orig, c_dq)
