"""The columnwise source and the identity direction of hybrid quantization
("Hybrid quantization", "Enable columnwise_source and hybrid recipes": with
columnwise_source="rowwise_dequantized" the backward operand is built from
dequantize(rowwise-quantized x), double quantization unless the columnwise
quantizer is the identity; IdentityQuantizer passes the high-precision value
through), GPU against the oracle bit for bit: rowwise codes, scales and
amax; the columnwise operand against the oracle's quantization of its own
dequantized rowwise value (or, for the identity, that value itself)."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import assert_codes_equal, assert_scales_equal, bits, qt_codes

pytestmark = pytest.mark.gpu
SIGN = inputs.rht_sign_vector()
DQ = nvq.COL_SOURCE_ROWWISE_DEQUANTIZED


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _x(M, K, seed):
    return inputs.normal_bf16((M, K), 1.0, torch.Generator().manual_seed(seed))


def _check_row(q, x, fmt, sr):
    xb = bits(x)
    if fmt == nvq.NVFP4:
        c, s, A = oracle.nvfp4_quantize_rows(xb, sr=sr)
        assert q.amax.item() == np.float32(A)
    elif fmt == nvq.MXFP8:
        c, s = oracle.mxfp8_quantize_rows(xb)
    else:
        assert np.array_equal(bits(q.bf16().cpu()), oracle.identity_rows(xb)), "identity rows"
        return
    assert_codes_equal(qt_codes(q), c, "row codes")
    assert_scales_equal(q, s, "row scales")


def _check_col(q, src_bits, fmt, rht, sr):
    """src_bits: the columnwise source (bf16 bits [M, K])."""
    if fmt == nvq.NVFP4:
        c, s, A = oracle.nvfp4_quantize_cols(src_bits, rht_sign=rht, sr=sr)
        assert q.amax.item() == np.float32(A), f"col amax {q.amax.item()} vs {A}"
    elif fmt == nvq.MXFP8:
        c, s = oracle.mxfp8_quantize_cols(src_bits)
    else:
        assert np.array_equal(bits(q.bf16().cpu()), oracle.identity_cols(src_bits)), "identity cols"
        return
    assert_codes_equal(qt_codes(q), c, "col codes")
    assert_scales_equal(q, s, "col scales")


SHAPES = [(256, 512), (300, 96), (40, 64), (129, 272)]
DQ_CASES = [  # (row, col, rht, sr)
    (nvq.NVFP4, nvq.MXFP8, False, False), (nvq.NVFP4, nvq.MXFP8, False, True),
    (nvq.NVFP4, nvq.NVFP4, False, False), (nvq.NVFP4, nvq.NVFP4, True, True),
    (nvq.MXFP8, nvq.NVFP4, True, False), (nvq.MXFP8, nvq.NVFP4, False, True),
    (nvq.MXFP8, nvq.MXFP8, False, False),
    (nvq.NVFP4, nvq.IDENTITY, False, False), (nvq.NVFP4, nvq.IDENTITY, False, True),
    (nvq.MXFP8, nvq.IDENTITY, False, False),
]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("row_fmt,col_fmt,rht,sr", DQ_CASES)
def test_rowwise_dequantized_source(M, K, row_fmt, col_fmt, rht, sr):
    if row_fmt == nvq.MXFP8 and K % 32:
        pytest.skip("MXFP8 rows need K % 32 == 0")
    x = _x(M, K, M * 3 + K)
    key = (4321, 2) if sr else None
    sign = SIGN if rht else None
    row, col = nvq.hybrid_quantize(x.cuda(), row_fmt, col_fmt, rht_sign=sign, sr=key, col_source=DQ)
    torch.cuda.synchronize()
    _check_row(row, x, row_fmt, key if row_fmt == nvq.NVFP4 else None)
    xd, _ = oracle.rowwise_dequantized(x, row_fmt, sr=key if row_fmt == nvq.NVFP4 else None)
    _check_col(col, xd, col_fmt, sign if col_fmt == nvq.NVFP4 else None, key if col_fmt == nvq.NVFP4 else None)


def test_rowwise_dequantized_identity_columnwise_matches_rowwise():
    """The review's test on the GPU: with the rowwise-dequantized source and an
    identity columnwise direction, the columnwise operand is the rowwise
    operand's dequantized value, transposed."""
    x = _x(256, 256, 9)
    for fmt in (nvq.NVFP4, nvq.MXFP8):
        row, col = nvq.hybrid_quantize(x.cuda(), fmt, nvq.IDENTITY, col_source=DQ)
        torch.cuda.synchronize()
        if fmt == nvq.NVFP4:
            c, s = qt_codes(row), oracle.scale_unswizzle(row.scale.cpu().numpy(), 256, 16)
            deq = oracle.nvfp4_dequant_bf16(c, s, row.amax.item())
        else:
            c, s = qt_codes(row), oracle.scale_unswizzle(row.scale.cpu().numpy(), 256, 8)
            deq = oracle.mxfp8_dequant_bf16(c, s)
        assert np.array_equal(bits(col.bf16().cpu()), deq.T)


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("row_fmt,col_fmt", [(nvq.NVFP4, nvq.IDENTITY), (nvq.NONE, nvq.IDENTITY),
                                             (nvq.IDENTITY, nvq.NONE), (nvq.IDENTITY, nvq.NVFP4),
                                             (nvq.IDENTITY, nvq.MXFP8), (nvq.MXFP8, nvq.IDENTITY)])
def test_identity_direction_original_source(M, K, row_fmt, col_fmt):
    if nvq.MXFP8 in (row_fmt,) and K % 32:
        pytest.skip("MXFP8 rows need K % 32 == 0")
    x = _x(M, K, M + 5 * K)
    sign = SIGN if col_fmt == nvq.NVFP4 else None
    row, col = nvq.hybrid_quantize(x.cuda(), row_fmt, col_fmt, rht_sign=sign)
    torch.cuda.synchronize()
    if row_fmt != nvq.NONE:
        _check_row(row, x, row_fmt, None)
    else:
        assert row is None
    if col_fmt != nvq.NONE:
        _check_col(col, bits(x), col_fmt, sign, None)
    else:
        assert col is None


def test_double_quantization_composes_two_quantizers():
    """The rowwise-dequantized NVFP4 -> MXFP8 columnwise operand equals the
    GPU's own MXFP8 columnwise quantization of the GPU's dequantized rowwise
    value (identity direction): the two-step pipeline and the fused call agree."""
    x = _x(512, 512, 10)
    _, fused = nvq.hybrid_quantize(x.cuda(), nvq.NVFP4, nvq.MXFP8, col_source=DQ)
    _, ident = nvq.hybrid_quantize(x.cuda(), nvq.NVFP4, nvq.IDENTITY, col_source=DQ)
    xd = ident.bf16().t().contiguous()
    _, two = nvq.mxfp8_quantize(xd, nvq.DIR_COL)
    torch.cuda.synchronize()
    assert torch.equal(fused.data, two.data) and torch.equal(fused.scale, two.scale)
