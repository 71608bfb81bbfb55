"""Grouped (MoE expert) quantize + GEMMs vs the oracle, per group.

"Hybrid quantization" (GroupedLinear, _hybrid_split_quantize, grouped GEMM):
forward with NVFP4 rowwise input/weight, dgrad and wgrad with MXFP8 operands
quantized columnwise from the original bf16, MXFP8 grad_output.  Empty groups
must work (a zero-length contraction gives a zero weight gradient).  The
grouped NVFP4 backward ("MXFP8 fwd and NVFP4 bwd (or vice versa)", with the
torchtitan recipe's SR on the gradient and RHT on the wgrad operands) is
checked with the stochastic-rounding index of each element at its position
in the padded grouped output."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import assert_codes_equal, assert_gemm_close, assert_scales_equal, bits, qt_codes

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


def _pad_starts(sizes):
    starts, p = [], 0
    for m in sizes:
        starts.append(p)
        p += -(-m // 128) * 128
    return starts, p


def _grouped_nvfp4_oracle(xb, sizes, rht=None, sr=None):
    """Oracle NVFP4 rows and columns of a grouped tensor in the padded layout:
    per group, its amaxes and its rows quantized at their padded positions.
    The columnwise direction quantizes the group's rows padded with zero rows
    to a multiple of 128, all of its 16-row blocks (with RHT a block of pad
    rows transforms to signed zeros, which keep their sign)."""
    K = xb.shape[1]
    starts, P = _pad_starts(sizes)
    rc = np.zeros((P, K // 2), np.uint8)
    rs = np.zeros((P, K // 16), np.uint8)
    cc = np.zeros((K, P // 2), np.uint8)
    cs = np.zeros((K, P // 16), np.uint8)
    ar = np.zeros(len(sizes), np.float32)
    ac = np.zeros(len(sizes), np.float32)
    src = 0
    for g, (m, p0) in enumerate(zip(sizes, starts)):
        if m:
            xg = xb[src:src + m]
            ar[g] = oracle.amax(xg)
            ac[g] = oracle.amax_rht_col(xg, rht) if rht is not None else oracle.amax(xg)
            c, sc = oracle.nvfp4_quantize_rows_at(xg, float(ar[g]), p0, sr=sr)
            rc[p0:p0 + m], rs[p0:p0 + m] = c, sc
            xp = np.zeros((-(-m // 128) * 128, K), np.uint16)
            xp[:m] = xg
            c, sc = oracle.nvfp4_quantize_cols_at(xp, float(ac[g]), p0, P, rht_sign=rht, sr=sr)
            cc[:, p0 // 2:p0 // 2 + c.shape[1]] = c
            cs[:, p0 // 16:p0 // 16 + sc.shape[1]] = sc
        src += m
    return (rc, rs, ar), (cc, cs, ac)


@pytest.mark.parametrize("rht,sr", [(True, True), (False, True), (True, False)])
def test_grouped_nvfp4_sr_rht_operands(rht, sr):
    """Grouped NVFP4 rows and columns with SR and / or RHT, bit for bit per
    group (amaxes, codes, swizzled scales), empty and ragged groups included."""
    x = inputs.student_t3_outliers(sum(SIZES), 256)
    sign = inputs.rht_sign_vector() if rht else None
    srv = (inputs.SR_SEED, 5) if sr else None
    xr, xc = nvq.grouped_hybrid_quantize(x.cuda(), SIZES, nvq.NVFP4, nvq.NVFP4, rht_sign=sign, sr=srv)
    torch.cuda.synchronize()
    (rc, rs, ar), (cc, cs, ac) = _grouped_nvfp4_oracle(bits(x), SIZES, sign, srv)
    assert np.array_equal(xr.amax.cpu().numpy(), ar), "row amaxes"
    assert np.array_equal(xc.amax.cpu().numpy(), ac), "column amaxes"
    assert_codes_equal(qt_codes(xr), rc, "grouped rows codes")
    assert_scales_equal(xr, rs, "grouped rows scales")
    assert_codes_equal(qt_codes(xc), cc, "grouped cols codes")
    assert_scales_equal(xc, cs, "grouped cols scales")


def test_grouped_nvfp4_backward_sr_rht():
    """A grouped NVFP4 backward: dgrad dx_g = dy_g W_g with dy SR-quantized,
    wgrad dW_g = dy_g^T x_g with both operands RHT'd (the transform cancels)
    and dy SR-quantized; each against the oracle's fp64 product of its own
    dequantized operands."""
    x, w, dy = _setup(SIZES)
    G, N, K = w.shape
    sign = inputs.rht_sign_vector()
    srv = (inputs.SR_SEED, 0)
    dyr, dyc = nvq.grouped_hybrid_quantize(dy.cuda(), SIZES, nvq.NVFP4, nvq.NVFP4, rht_sign=sign, sr=srv)
    _, xc = nvq.grouped_hybrid_quantize(x.cuda(), SIZES, nvq.NONE, nvq.NVFP4, rht_sign=sign)
    _, wc = nvq.grouped_hybrid_quantize(w.reshape(G * N, K).cuda(), [N] * G, nvq.NONE, nvq.NVFP4)
    dx = nvq.grouped_gemm_rows(dyr, wc, SIZES, N, b_col_groups=True)
    dw = nvq.grouped_gemm_wgrad(dyc, xc, SIZES)
    torch.cuda.synchronize()
    (drc, drs, dar), (dcc, dcs, dac) = _grouped_nvfp4_oracle(bits(dy), SIZES, sign, srv)
    _, (xcc, xcs, xac) = _grouped_nvfp4_oracle(bits(x), SIZES, sign, None)
    assert_codes_equal(qt_codes(dyr), drc, "dy rows codes")
    assert_codes_equal(qt_codes(dyc), dcc, "dy cols codes")
    assert_codes_equal(qt_codes(xc), xcc, "x cols codes")
    starts, P = _pad_starts(SIZES)
    wb = bits(w)
    src = 0
    for g, (m, p0) in enumerate(zip(SIZES, starts)):
        if m == 0:
            assert torch.count_nonzero(dw[g]).item() == 0
            continue
        wcc, wcs, wa = oracle.nvfp4_quantize_cols(wb[g])  # [K][N]
        a = oracle.nvfp4_dequant(drc[p0:p0 + m], drs[p0:p0 + m], oracle.nvfp4_g(float(dar[g])))
        assert_gemm_close(dx[src:src + m], oracle.gemm_tn_f64(a, oracle.nvfp4_dequant(wcc, wcs, oracle.nvfp4_g(wa))),
                          f"group {g} dgrad")
        mp = -(-m // 128) * 128
        da = oracle.nvfp4_dequant(dcc[:, p0 // 2:(p0 + mp) // 2], dcs[:, p0 // 16:(p0 + mp) // 16],
                                  oracle.nvfp4_g(float(dac[g])))
        xa = oracle.nvfp4_dequant(xcc[:, p0 // 2:(p0 + mp) // 2], xcs[:, p0 // 16:(p0 + mp) // 16],
                                  oracle.nvfp4_g(float(xac[g])))
        # a group of fewer than 16 tokens contracts over one Hadamard block:
        # every output is a short sum with heavy cancellation, so a few more
        # elements land 2 bf16 ulps from the fp64 value (the Frobenius bar holds)
        assert_gemm_close(dw[g], oracle.gemm_tn_f64(da, xa), f"group {g} wgrad", ulp_frac=0.999 if m >= 16 else 0.99)
        src += m
