"""Grouped (MoE expert) quantize + GEMMs vs the oracle, per group.

"Hybrid quantization" (GroupedLinear, _hybrid_split_quantize, grouped GEMM):
forward with NVFP4 rowwise input/weight, dgrad and wgrad with MXFP8 operands
quantized columnwise from the original bf16, MXFP8 grad_output.  Empty groups
must work (a zero-length contraction gives a zero weight gradient)."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import assert_gemm_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _randn(shape, seed, std=1.0):
    return inputs.normal_bf16(shape, std, torch.Generator().manual_seed(seed))


SIZES = [130, 0, 5, 256, 0, 77, 1]


def _setup(sizes, K=256, N=128):
    G = len(sizes)
    x = _randn((sum(sizes), K), 1)
    w = _randn((G, N, K), 2, 0.02)
    dy = _randn((sum(sizes), N), 3, 0.01)
    return x, w, dy


def test_grouped_forward_nvfp4():
    x, w, _ = _setup(SIZES)
    G, N, K = w.shape
    xr, _ = nvq.grouped_hybrid_quantize(x.cuda(), SIZES, nvq.NVFP4, nvq.NONE)
    wr, _ = nvq.grouped_hybrid_quantize(w.reshape(G * N, K).cuda(), [N] * G, nvq.NVFP4, nvq.NONE)
    y = nvq.grouped_gemm_rows(xr, wr, SIZES, N, b_col_groups=False)
    torch.cuda.synchronize()
    xb, wb = bits(x), bits(w)
    src = 0
    for g, m in enumerate(SIZES):
        if m:
            ac, asc, Aa = oracle.nvfp4_quantize_rows(xb[src:src + m])
            bc, bsc, Ab = oracle.nvfp4_quantize_rows(wb[g])
            ref = oracle.gemm_tn_f64(oracle.nvfp4_dequant(ac, asc, oracle.nvfp4_g(Aa)),
                                     oracle.nvfp4_dequant(bc, bsc, oracle.nvfp4_g(Ab)))
            assert_gemm_close(y[src:src + m], ref, f"group {g} fwd")
        src += m


def test_grouped_dgrad_mxfp8():
    """dx_g = dy_g W_g: A = dy rowwise MXFP8, B = W_g columnwise MXFP8 ([K][G*N])."""
    x, w, dy = _setup(SIZES)
    G, N, K = w.shape
    dyr, _ = nvq.grouped_hybrid_quantize(dy.cuda(), SIZES, nvq.MXFP8, nvq.NONE)
    _, wc = nvq.grouped_hybrid_quantize(w.reshape(G * N, K).cuda(), [N] * G, nvq.NONE, nvq.MXFP8)
    dx = nvq.grouped_gemm_rows(dyr, wc, SIZES, N, b_col_groups=True)
    torch.cuda.synchronize()
    dyb, wb = bits(dy), bits(w)
    src = 0
    for g, m in enumerate(SIZES):
        if m:
            ac, asc = oracle.mxfp8_quantize_rows(dyb[src:src + m])
            bc, bsc = oracle.mxfp8_quantize_cols(wb[g])  # [K][N]
            ref = oracle.gemm_tn_f64(oracle.mxfp8_dequant(ac, asc), oracle.mxfp8_dequant(bc, bsc))
            assert_gemm_close(dx[src:src + m], ref, f"group {g} dgrad")
        src += m


def test_grouped_wgrad_mxfp8_with_empty_groups():
    """dW_g = dy_g^T x_g over the group's (128-padded) tokens; empty groups -> 0."""
    x, w, dy = _setup(SIZES)
    G, N, K = w.shape
    _, dyc = nvq.grouped_hybrid_quantize(dy.cuda(), SIZES, nvq.NONE, nvq.MXFP8)
    _, xc = nvq.grouped_hybrid_quantize(x.cuda(), SIZES, nvq.NONE, nvq.MXFP8)
    dw = nvq.grouped_gemm_wgrad(dyc, xc, SIZES)
    torch.cuda.synchronize()
    xb, dyb = bits(x), bits(dy)
    src = 0
    for g, m in enumerate(SIZES):
        if m == 0:
            assert torch.count_nonzero(dw[g]).item() == 0
            continue
        mp = -(-m // 128) * 128
        xp = np.zeros((mp, K), np.uint16); xp[:m] = xb[src:src + m]
        dp = np.zeros((mp, N), np.uint16); dp[:m] = dyb[src:src + m]
        ac, asc = oracle.mxfp8_quantize_cols(dp)
        bc, bsc = oracle.mxfp8_quantize_cols(xp)
        ref = oracle.gemm_tn_f64(oracle.mxfp8_dequant(ac, asc), oracle.mxfp8_dequant(bc, bsc))
        assert_gemm_close(dw[g], ref, f"group {g} wgrad")
        src += m


def test_all_groups_empty():
    sizes = [0, 0, 0]
    x = torch.zeros(0, 256, dtype=torch.bfloat16)
    dy = torch.zeros(0, 128, dtype=torch.bfloat16)
    _, dyc = nvq.grouped_hybrid_quantize(dy.cuda(), sizes, nvq.NONE, nvq.MXFP8)
    _, xc = nvq.grouped_hybrid_quantize(x.cuda(), sizes, nvq.NONE, nvq.MXFP8)
    dw = nvq.grouped_gemm_wgrad(dyc, xc, sizes)
    torch.cuda.synchronize()
    assert dw.shape == (3, 128, 256) and torch.count_nonzero(dw).item() == 0
