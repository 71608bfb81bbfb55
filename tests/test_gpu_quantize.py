"""GPU quantizers vs the CPU oracle: codes, swizzled scales and amax must be
bit-identical (including stochastic rounding under the same Philox stream and
the Hadamard transform), through the C ABI.

Pages: "Add an NVFP4 quantization converter" (NVFP4 block quantization, RHT,
SR) and "Hybrid quantization" (MXFP8, per-direction hybrid formats, grouped
split quantization, ceil(M/32) columnwise scales)."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import (bits, check_mxfp8_col, check_mxfp8_row, check_nvfp4_col, check_nvfp4_row, qt_codes,
                      qt_scales, assert_codes_equal, assert_scales_equal)

pytestmark = pytest.mark.gpu
SIGN = inputs.rht_sign_vector()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _randn(M, K, seed=0, std=1.0):
    return inputs.normal_bf16((M, K), std, torch.Generator().manual_seed(seed))


SHAPES = [(256, 512), (40, 64), (1, 16), (300, 48), (129, 272), (128, 256)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_nvfp4_rows_rtn(M, K):
    x = _randn(M, K, seed=M + K)
    row, _ = nvq.nvfp4_quantize(x.cuda(), nvq.DIR_ROW)
    torch.cuda.synchronize()
    check_nvfp4_row(row, x)


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("rht,sr", [(False, False), (True, False), (False, True), (True, True)])
def test_nvfp4_rows_and_cols(M, K, rht, sr):
    x = _randn(M, K, seed=3 * M + K)
    sign = SIGN if rht else None
    key = (1234, 0) if sr else None
    row, col = nvq.nvfp4_quantize(x.cuda(), nvq.DIR_ROW | nvq.DIR_COL, rht_sign=sign, sr=key)
    torch.cuda.synchronize()
    check_nvfp4_row(row, x, sr=key)
    check_nvfp4_col(col, x, rht=sign, sr=key)


def test_nvfp4_sr_offset_and_negative_seed():
    x = _randn(64, 128, seed=9)
    key = (-(2 ** 63) + 12345, 7)
    row, col = nvq.nvfp4_quantize(x.cuda(), 3, rht_sign=SIGN, sr=key)
    torch.cuda.synchronize()
    check_nvfp4_row(row, x, sr=key)
    check_nvfp4_col(col, x, rht=SIGN, sr=key)


@pytest.mark.parametrize("M,K", [(256, 512), (48, 64), (33, 32), (1, 32), (300, 96)])
def test_mxfp8_rows_and_cols(M, K):
    x = _randn(M, K, seed=M * 7 + K)
    row, col = nvq.mxfp8_quantize(x.cuda(), nvq.DIR_ROW | nvq.DIR_COL)
    torch.cuda.synchronize()
    check_mxfp8_row(row, x)
    check_mxfp8_col(col, x)
    assert col.cols == -(-M // 32) * 32  # ceil, not floor


def test_mxfp8_cols_only_ragged_k():
    x = _randn(70, 80, seed=4)  # K not a multiple of 32 is fine for the columnwise direction
    _, col = nvq.mxfp8_quantize(x.cuda(), nvq.DIR_COL)
    torch.cuda.synchronize()
    check_mxfp8_col(col, x)


@pytest.mark.parametrize("row_fmt,col_fmt", [(1, 2), (2, 1), (1, 0), (0, 2), (2, 2), (1, 1)])
def test_hybrid_matches_single_format_oracle(row_fmt, col_fmt):
    x = _randn(192, 256, seed=11)
    sign = SIGN if col_fmt == 1 else None
    row, col = nvq.hybrid_quantize(x.cuda(), row_fmt, col_fmt, rht_sign=sign)
    torch.cuda.synchronize()
    if row_fmt == 1:
        check_nvfp4_row(row, x)
    elif row_fmt == 2:
        check_mxfp8_row(row, x)
    else:
        assert row is None
    if col_fmt == 1:
        check_nvfp4_col(col, x, rht=sign)
    elif col_fmt == 2:
        check_mxfp8_col(col, x)
    else:
        assert col is None


@pytest.mark.parametrize("fmt", [1, 2])
def test_hybrid_same_format_is_bitwise_base_recipe(fmt):
    """hybrid(X, X) == X bitwise ("Hybrid quantization": hybrid vs vanilla recipe parity)."""
    x = _randn(256, 256, seed=12).cuda()
    hr, hc = nvq.hybrid_quantize(x, fmt, fmt)
    br, bc = (nvq.nvfp4_quantize(x, 3) if fmt == 1 else nvq.mxfp8_quantize(x, 3))
    torch.cuda.synchronize()
    for a, b in ((hr, br), (hc, bc)):
        assert torch.equal(a.data, b.data) and torch.equal(a.scale, b.scale)
        if fmt == 1:
            assert torch.equal(a.amax, b.amax)


def test_edge_values():
    """zeros, signed zeros, tiny and huge magnitudes, a zero tensor.  Values up
    to 3e38 go through the paths without the Hadamard transform; with it, the
    magnitudes stay below FLT_MAX / 16 so the fp32 butterfly cannot overflow
    (inputs whose transform overflows are outside the defined domain)."""
    def table(big):
        vals = torch.tensor([0.0, -0.0, 1e-30, -1e-30, big, -big, 1.0, -2.5, 6.0, 448.0, 1e-40],
                            dtype=torch.float32)
        return vals.repeat(64 * 64 // vals.numel() + 1)[: 64 * 64].reshape(64, 64).to(torch.bfloat16)

    for big in (3e38, 2e37):
        x = table(big)
        for t in (x, torch.zeros(64, 64, dtype=torch.bfloat16), x * 0 - 0.0):
            rht = SIGN if big < 1e38 else None
            row, col = nvq.nvfp4_quantize(t.cuda(), 3, rht_sign=rht, sr=(5, 0))
            mr, mc = nvq.mxfp8_quantize(t.cuda(), 3)
            torch.cuda.synchronize()
            check_nvfp4_row(row, t, sr=(5, 0))
            check_nvfp4_col(col, t, rht=rht, sr=(5, 0))
            check_mxfp8_row(mr, t)
            check_mxfp8_col(mc, t)


def test_rht_overflow_is_what_the_header_says():
    """Outside the stated domain: |x| close to FLT_MAX makes the fp32 butterfly
    of the columnwise Hadamard transform overflow.  nvq.h says the call then
    completes with no device error, the columnwise amax is +inf, and the
    rowwise direction (no transform) is unaffected -- bit-exact here."""
    vals = torch.tensor([3e38, 3e38, -3e38, 1.0, -2.5, 0.0, 448.0, 1e-30], dtype=torch.float32)
    x = vals.repeat(64 * 64 // vals.numel())[: 64 * 64].reshape(64, 64).to(torch.bfloat16)
    assert np.isinf(oracle.amax_rht_col(bits(x), SIGN))  # the transform does overflow
    row, col = nvq.nvfp4_quantize(x.cuda(), 3, rht_sign=SIGN, sr=(5, 0))
    torch.cuda.synchronize()
    assert nvq.device_status() == 0
    a = col.amax.item()
    assert np.isinf(a) and a > 0
    check_nvfp4_row(row, x, sr=(5, 0))


def test_amax_entry_point():
    x = inputs.student_t3_outliers(512, 256)
    a, r = nvq.amax(x.cuda(), rht_sign=SIGN)
    torch.cuda.synchronize()
    assert a.item() == np.float32(oracle.amax(bits(x)))
    assert r.item() == np.float32(oracle.amax_rht_col(bits(x), SIGN))


def test_strided_input():
    base = _randn(128, 384, seed=13)
    x = base[:, 64:320]  # ld = 384 > K = 256
    xd = base.cuda()[:, 64:320]
    row, col = nvq.nvfp4_quantize(xd, 3, rht_sign=SIGN)
    torch.cuda.synchronize()
    check_nvfp4_row(row, x.contiguous())
    check_nvfp4_col(col, x.contiguous(), rht=SIGN)


def _grouped_oracle_rows(x, sizes, fmt):
    """Oracle per-group quantization assembled into the padded layout."""
    xb = bits(x)
    K = xb.shape[1]
    P = sum(-(-m // 128) * 128 for m in sizes)
    per_row = K // 2 if fmt == 1 else K
    blk = 16 if fmt == 1 else 32
    codes = np.zeros((P, per_row), np.uint8)
    scales = np.zeros((P, K // blk), np.uint8)
    amax = []
    src = dst = 0
    for m in sizes:
        if m:
            if fmt == 1:
                c, s, A = oracle.nvfp4_quantize_rows(xb[src:src + m])
            else:
                (c, s), A = oracle.mxfp8_quantize_rows(xb[src:src + m]), 0.0
            codes[dst:dst + m], scales[dst:dst + m] = c, s
        else:
            A = 0.0
        amax.append(A)
        src += m
        dst += -(-m // 128) * 128
    return codes, scales, amax


def _grouped_oracle_cols(x, sizes, fmt):
    xb = bits(x)
    K = xb.shape[1]
    P = sum(-(-m // 128) * 128 for m in sizes)
    blk = 16 if fmt == 1 else 32
    codes = np.zeros((K, P // 2 if fmt == 1 else P), np.uint8)
    scales = np.zeros((K, P // blk), np.uint8)
    amax = []
    src = dst = 0
    for m in sizes:
        mp = -(-m // 128) * 128
        if m:
            pad = np.zeros((mp, K), np.uint16)
            pad[:m] = xb[src:src + m]
            if fmt == 1:
                c, s, A = oracle.nvfp4_quantize_cols(pad)
                codes[:, dst // 2:(dst + mp) // 2] = c
            else:
                c, s = oracle.mxfp8_quantize_cols(pad)
                A = 0.0
                codes[:, dst:dst + mp] = c
            scales[:, dst // blk:(dst + mp) // blk] = s
        else:
            A = 0.0
        amax.append(A)
        src += m
        dst += mp
    return codes, scales, amax


@pytest.mark.parametrize("row_fmt,col_fmt", [(1, 2), (2, 2), (1, 1), (2, 1)])
def test_grouped_hybrid_quantize(row_fmt, col_fmt):
    sizes = [5, 0, 130, 1, 0, 256, 77]
    K = 256
    x = _randn(sum(sizes), K, seed=21)
    row, col = nvq.grouped_hybrid_quantize(x.cuda(), sizes, row_fmt, col_fmt)
    torch.cuda.synchronize()
    rc, rs, ra = _grouped_oracle_rows(x, sizes, row_fmt)
    assert_codes_equal(qt_codes(row), rc, "grouped row codes")
    assert_scales_equal(row, rs, "grouped row scales")
    cc, cs, ca = _grouped_oracle_cols(x, sizes, col_fmt)
    assert_codes_equal(qt_codes(col), cc, "grouped col codes")
    assert_scales_equal(col, cs, "grouped col scales")
    if row_fmt == 1:
        assert np.array_equal(row.amax.cpu().numpy(), np.array(ra, np.float32))
    if col_fmt == 1:
        assert np.array_equal(col.amax.cpu().numpy(), np.array(ca, np.float32))


@pytest.mark.parametrize("M", [2048, 8192])
def test_quant_sweep_sizes_bit_exact(M):
    """The quantize-sweep workload (0.1*t(3), 0.1% outlier channels), all variants."""
    x = inputs.student_t3_outliers(M)
    xd = x.cuda()
    r1, c1 = nvq.nvfp4_quantize(xd, 3)
    r2, c2 = nvq.nvfp4_quantize(xd, 3, rht_sign=SIGN, sr=(inputs.SR_SEED, 0))
    r3, c3 = nvq.mxfp8_quantize(xd, 3)
    torch.cuda.synchronize()
    check_nvfp4_row(r1, x)
    check_nvfp4_col(c1, x)
    check_nvfp4_row(r2, x, sr=(inputs.SR_SEED, 0))
    check_nvfp4_col(c2, x, rht=SIGN, sr=(inputs.SR_SEED, 0))
    check_mxfp8_row(r3, x)
    check_mxfp8_col(c3, x)
