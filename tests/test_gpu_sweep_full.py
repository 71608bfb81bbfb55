"""The quantize sweep's largest tensor, x[131072, 4096] (0.1 * Student-t(3)
with 0.1% outlier channels), in the launch configuration the benchmark times:
NVFP4 row + col round-to-nearest, NVFP4 row + col with the Hadamard transform
on the columnwise copy and stochastic rounding on both, and MXFP8 row + col.

The oracle reads the whole tensor for the amaxes (plain and Hadamard-domain),
then quantizes sampled row ranges -- the first, two interior and the last --
as rows of the whole tensor (same amax, same Philox counters), and those rows
and contraction columns of the GPU outputs must match it bit for bit (codes
and scales).  The grid is 16 x 1024 CTAs, so the ranges span distant CTAs.

Pages: "Add an NVFP4 quantization converter" (NVFP4, RHT, SR) and "Hybrid
quantization" (MXFP8, ceil(M/32) columnwise scales)."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import assert_codes_equal, bits, qt_codes, qt_scales

pytestmark = pytest.mark.gpu

M = 131072
RANGES = ((0, 256), (40960, 160), (90112, 288), (M - 256, 256))  # (first row, rows): multiples of 32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _row_scales(q, r0, n):
    """Compact scales of rows [r0, r0 + n) from the swizzled buffer (whole
    128-row tiles are read and un-swizzled)."""
    blk = 16 if q.fmt == nvq.NVFP4 else 32
    nb = q.cols // blk
    t0, t1 = r0 // 128, -(-(r0 + n) // 128)
    ct = -(-nb // 4)
    buf = qt_scales(q)[t0 * ct * 512:t1 * ct * 512]
    comp = oracle.scale_unswizzle(buf, (t1 - t0) * 128, nb)
    return comp[r0 - t0 * 128:r0 - t0 * 128 + n]


def _check_nvfp4(row, col, xb, sign, sr):
    K = xb.shape[1]
    A = oracle.amax(xb)
    A_col = oracle.amax_rht_col(xb, sign) if sign is not None else A
    assert row.amax.item() == np.float32(A)
    assert col.amax.item() == np.float32(A_col)
    rc, cc = qt_codes(row), qt_codes(col)
    cs = oracle.scale_unswizzle(qt_scales(col), K, M // 16)
    for r0, n in RANGES:
        c, s = oracle.nvfp4_quantize_rows_at(xb[r0:r0 + n], A, r0, sr=sr)
        assert_codes_equal(rc[r0:r0 + n], c, f"rows {r0}+{n} codes")
        assert np.array_equal(_row_scales(row, r0, n), s), f"rows {r0}+{n} scales"
        c, s = oracle.nvfp4_quantize_cols_at(xb[r0:r0 + n], A_col, r0, M, rht_sign=sign, sr=sr)
        assert_codes_equal(cc[:, r0 // 2:(r0 + n) // 2], c, f"cols {r0}+{n} codes")
        assert np.array_equal(cs[:, r0 // 16:(r0 + n) // 16], s), f"cols {r0}+{n} scales"


def test_quant_sweep_131072_sampled_bit_exact():
    x = inputs.student_t3_outliers(M)
    xb = bits(x)
    K = xb.shape[1]
    xd = x.cuda()
    del x
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)

    r, c = nvq.nvfp4_quantize(xd, 3)
    torch.cuda.synchronize()
    _check_nvfp4(r, c, xb, None, None)
    del r, c

    r, c = nvq.nvfp4_quantize(xd, 3, rht_sign=sign, sr=sr)
    torch.cuda.synchronize()
    _check_nvfp4(r, c, xb, sign, sr)
    del r, c

    r, c = nvq.mxfp8_quantize(xd, 3)
    torch.cuda.synchronize()
    assert c.cols == M
    rc, cc = qt_codes(r), qt_codes(c)
    cs = oracle.scale_unswizzle(qt_scales(c), K, M // 32)
    for r0, n in RANGES:
        codes, scales = oracle.mxfp8_quantize_rows(xb[r0:r0 + n])
        assert_codes_equal(rc[r0:r0 + n], codes, f"mxfp8 rows {r0}+{n} codes")
        assert np.array_equal(_row_scales(r, r0, n), scales), f"mxfp8 rows {r0}+{n} scales"
        codes, scales = oracle.mxfp8_quantize_cols(xb[r0:r0 + n])
        assert_codes_equal(cc[:, r0:r0 + n], codes, f"mxfp8 cols {r0}+{n} codes")
        assert np.array_equal(cs[:, r0 // 32:(r0 + n) // 32], scales), f"mxfp8 cols {r0}+{n} scales"
