"""NVFP4 2D (16 x 16) columnwise block scaling and the linear layer with
per-direction formats, GPU against the oracle ("Hybrid quantization": the
timeline's "[Common] Enable NVFP4 2D block scaling in columnwise only", and
the Description's "MXFP8 fwd and NVFP4 bwd (or vice versa)").  Quantized
operands bit for bit; GEMM outputs within the GEMM tolerance of the oracle's
fp64 product of its own operands."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import (assert_codes_equal, assert_gemm_close, assert_scales_equal, bits, check_mxfp8_col,
                      check_mxfp8_row, check_nvfp4_col, check_nvfp4_row)

pytestmark = pytest.mark.gpu
SIGN = inputs.rht_sign_vector()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _check_2d(q, x, what="2D col"):
    c, s, A = oracle.nvfp4_quantize_cols_2d(bits(x))
    assert q.amax.item() == np.float32(A), what + " amax"
    assert_codes_equal(q.data[: c.size].cpu().numpy().reshape(c.shape), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s, A


@pytest.mark.parametrize("M,K", [(256, 512), (300, 96), (40, 64), (129, 272)])
@pytest.mark.parametrize("row_fmt", [nvq.NONE, nvq.NVFP4, nvq.MXFP8])
def test_nvfp4_2d_columnwise(M, K, row_fmt):
    if row_fmt == nvq.MXFP8 and K % 32:
        pytest.skip("MXFP8 rows need K % 32 == 0")
    x = inputs.student_t3_outliers(M, K)
    row, col = nvq.hybrid_quantize(x.cuda(), row_fmt, nvq.NVFP4, col_2d=True)
    torch.cuda.synchronize()
    _check_2d(col, x)
    if row_fmt == nvq.NVFP4:
        check_nvfp4_row(row, x)
    elif row_fmt == nvq.MXFP8:
        check_mxfp8_row(row, x)


def _deq(fmt, t):
    if fmt == nvq.NVFP4:
        c, s, A = t
        return oracle.nvfp4_dequant(c, s, oracle.nvfp4_g(A))
    c, s = t[:2]
    return oracle.mxfp8_dequant(c, s)


@pytest.mark.parametrize("fwd_fmt,bwd_fmt,w2d", [(nvq.MXFP8, nvq.NVFP4, True), (nvq.MXFP8, nvq.NVFP4, False),
                                                  (nvq.NVFP4, nvq.MXFP8, False)])
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (512, 256, 256)])
def test_hybrid_linear_recipe(fwd_fmt, bwd_fmt, w2d, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    x = inputs.normal_bf16((M, K), 1.0, g)
    w = inputs.normal_bf16((N, K), 0.02, g)
    dy = inputs.normal_bf16((M, N), 0.01, g)
    sr = (inputs.SR_SEED, 0)
    nv_bwd = bwd_fmt == nvq.NVFP4
    y, saved = nvq.hybrid_linear_fwd(x.cuda(), w.cuda(), fwd_fmt, bwd_fmt, rht_sign=SIGN, w_col_2d=w2d)
    bw = nvq.hybrid_linear_bwd_quantize(dy.cuda(), bwd_fmt, rht_sign=SIGN, sr=sr)
    dx = nvq.linear_dgrad(bw["dy_row"], saved["w_col"])
    dw = nvq.linear_wgrad(bw["dy_col"], saved["x_col"])
    torch.cuda.synchronize()
    # forward operands
    if fwd_fmt == nvq.NVFP4:
        xr, wr = check_nvfp4_row(saved["x_row"], x), check_nvfp4_row(saved["w_row"], w)
    else:
        xr, wr = check_mxfp8_row(saved["x_row"], x), check_mxfp8_row(saved["w_row"], w)
    # backward operands
    if nv_bwd:
        xc = check_nvfp4_col(saved["x_col"], x, rht=SIGN)
        wc = _check_2d(saved["w_col"], w, "W col 2D") if w2d else check_nvfp4_col(saved["w_col"], w)
        dr = check_nvfp4_row(bw["dy_row"], dy, sr=sr)
        dc = check_nvfp4_col(bw["dy_col"], dy, rht=SIGN, sr=sr)
    else:
        xc, wc = check_mxfp8_col(saved["x_col"], x), check_mxfp8_col(saved["w_col"], w)
        dr, dc = check_mxfp8_row(bw["dy_row"], dy), check_mxfp8_col(bw["dy_col"], dy)
    assert_gemm_close(y, oracle.gemm_tn_f64(_deq(fwd_fmt, xr), _deq(fwd_fmt, wr)), "fwd")
    assert_gemm_close(dx, oracle.gemm_tn_f64(_deq(bwd_fmt, dr), _deq(bwd_fmt, wc)), "dgrad")
    assert_gemm_close(dw, oracle.gemm_tn_f64(_deq(bwd_fmt, dc), _deq(bwd_fmt, xc)), "wgrad")
