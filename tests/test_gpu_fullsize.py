"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times.

* Llama-3-8B MLP up-projection (x[16384,4096], W[14336,4096], dy[16384,14336],
  SR seed 1234, RHT signs seed 7): every quantized operand of the step is
  compared bit for bit with the oracle over the whole tensor; the three GEMM
  outputs on sampled entries (random positions plus one full row and one full
  column) that the oracle computes one by one from its own operands.
* MoE grouped linear (64 experts 4096->1536, 65536 Zipf(1.1) tokens): operands
  and outputs of a spread of experts (the smallest, the largest, empty ones)
  against the oracle.

Pages: "Add an NVFP4 quantization converter" (Llama-3-8B run, NVFP4Linear) and
"Hybrid quantization" (GroupedLinear with NVFP4 forward / MXFP8 backward)."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import (assert_codes_equal, assert_scales_equal, bits, check_sampled_gemm, qt_codes, qt_scales,
                      sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


_sample_positions = sample_positions
_check_sampled = check_sampled_gemm


def test_llama3_8b_up_step_full_size():
    M, N, K = inputs.LLAMA3_8B_UP["M"], inputs.LLAMA3_8B_UP["N"], inputs.LLAMA3_8B_UP["K"]
    x, w, dy = inputs.llama_up()
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    y, saved = nvq.nvfp4_linear_fwd(x.cuda(), w.cuda(), rht_sign=sign)
    bw = nvq.nvfp4_linear_bwd_quantize(dy.cuda(), rht_sign=sign, sr=sr)
    dx = nvq.nvfp4_linear_dgrad(bw["dy_row"], saved["w_col"])
    dw = nvq.nvfp4_linear_wgrad(bw["dy_col"], saved["x_col"])
    torch.cuda.synchronize()

    xb, wb, dyb = bits(x), bits(w), bits(dy)
    ops = {
        "x_row": (saved["x_row"], oracle.nvfp4_quantize_rows(xb)),
        "x_col": (saved["x_col"], oracle.nvfp4_quantize_cols(xb, rht_sign=sign)),
        "w_row": (saved["w_row"], oracle.nvfp4_quantize_rows(wb)),
        "w_col": (saved["w_col"], oracle.nvfp4_quantize_cols(wb)),
        "dy_row": (bw["dy_row"], oracle.nvfp4_quantize_rows(dyb, sr=sr)),
        "dy_col": (bw["dy_col"], oracle.nvfp4_quantize_cols(dyb, rht_sign=sign, sr=sr)),
    }
    for name, (q, (c, s, A)) in ops.items():
        assert q.amax.item() == np.float32(A), name
        assert_codes_equal(qt_codes(q), c, name + " codes")
        assert_scales_equal(q, s, name + " scales")

    _check_sampled(y.cpu(), 1, ops["x_row"][1], ops["w_row"][1], K, *_sample_positions(M, N, 4096, 1), "fwd y")
    _check_sampled(dx.cpu(), 1, ops["dy_row"][1], ops["w_col"][1], N, *_sample_positions(M, K, 4096, 2), "dgrad dx")
    _check_sampled(dw.cpu(), 1, ops["dy_col"][1], ops["x_col"][1], M, *_sample_positions(N, K, 4096, 3), "wgrad dW")


def test_moe_grouped_full_size():
    sizes, x, w, dy = inputs.moe_grouped()
    G, Nn, K = w.shape
    sizes = [int(v) for v in sizes]
    xr, xc = nvq.grouped_hybrid_quantize(x.cuda(), sizes, nvq.NVFP4, nvq.MXFP8)
    wr, wc = nvq.grouped_hybrid_quantize(w.reshape(G * Nn, K).cuda(), [Nn] * G, nvq.NVFP4, nvq.MXFP8)
    dyr, dyc = nvq.grouped_hybrid_quantize(dy.cuda(), sizes, nvq.MXFP8, nvq.MXFP8)
    y = nvq.grouped_gemm_rows(xr, wr, sizes, Nn, b_col_groups=False)
    dx = nvq.grouped_gemm_rows(dyr, wc, sizes, Nn, b_col_groups=True)
    dw = nvq.grouped_gemm_wgrad(dyc, xc, sizes)
    torch.cuda.synchronize()
    assert y.shape == (sum(sizes), Nn) and dx.shape == (sum(sizes), K) and dw.shape == (G, Nn, K)

    order = np.argsort(sizes)
    picks = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[len(order) // 2]), 5, 40]))
    offs = np.concatenate([[0], np.cumsum(sizes)])
    poffs = np.concatenate([[0], np.cumsum([-(-m // 128) * 128 for m in sizes])])
    P = int(poffs[-1])
    xb, wb, dyb = bits(x), bits(w), bits(dy)
    xr_c, dyr_c, wr_c = qt_codes(xr), qt_codes(dyr), qt_codes(wr)
    xc_c, wc_c, dyc_c = qt_codes(xc), qt_codes(wc), qt_codes(dyc)
    # columnwise MXFP8 scales in compact form (the columns of one expert are not
    # whole scale tiles, so the swizzled buffers are read back whole)
    xc_s = oracle.scale_unswizzle(qt_scales(xc), K, P // 32)
    wc_s = oracle.scale_unswizzle(qt_scales(wc), K, G * Nn // 32)
    dyc_s = oracle.scale_unswizzle(qt_scales(dyc), Nn, P // 32)

    def rows_scales(q, r0, rows, compact, what):
        """Swizzled scales of whole 128-row tiles [r0, r0 + rows) against the
        oracle's compact scales (zero-padded to the tiles)."""
        blk = 16 if q.fmt == nvq.NVFP4 else 32
        nb = q.cols // blk
        pad = np.zeros((rows, nb), np.uint8)
        pad[:compact.shape[0]] = compact
        want = oracle.scale_swizzle(pad)
        t0 = (r0 // 128) * (-(-nb // 4)) * 512
        got = qt_scales(q)[t0:t0 + want.size]
        assert np.array_equal(got, want), what

    for g in picks:
        m, s0, p0 = sizes[g], int(offs[g]), int(poffs[g])
        mp = -(-m // 128) * 128
        # the expert's weights in both formats (every expert has N rows)
        b = oracle.nvfp4_quantize_rows(wb[g])
        assert_codes_equal(wr_c[g * Nn:(g + 1) * Nn], b[0], f"expert {g} w_row codes")
        rows_scales(wr, g * Nn, Nn, b[1], f"expert {g} w_row scales")
        db = oracle.mxfp8_quantize_cols(wb[g]) + (0.0,)
        assert_codes_equal(wc_c[:, g * Nn:(g + 1) * Nn], db[0], f"expert {g} w_col codes")
        assert np.array_equal(wc_s[:, g * Nn // 32:(g + 1) * Nn // 32], db[1]), f"expert {g} w_col scales"
        if m == 0:
            assert torch.count_nonzero(dw[g]).item() == 0
            continue
        # forward operands (NVFP4 rows) and output
        a = oracle.nvfp4_quantize_rows(xb[s0:s0 + m])
        assert_codes_equal(xr_c[p0:p0 + m], a[0], f"expert {g} x_row codes")
        assert not xr_c[p0 + m:p0 + mp].any(), f"expert {g} x_row pad rows"
        rows_scales(xr, p0, mp, a[1], f"expert {g} x_row scales")
        assert xr.amax[g].item() == np.float32(a[2]) and wr.amax[g].item() == np.float32(b[2])
        rows, cols = _sample_positions(m, Nn, 512, 10 + g)
        _check_sampled(y[s0:s0 + m].cpu(), 1, a, b, K, rows, cols, f"expert {g} fwd")
        # dgrad: MXFP8 dy rows x MXFP8 W columns
        da = oracle.mxfp8_quantize_rows(dyb[s0:s0 + m]) + (0.0,)
        assert_codes_equal(dyr_c[p0:p0 + m], da[0], f"expert {g} dy_row codes")
        rows_scales(dyr, p0, mp, da[1], f"expert {g} dy_row scales")
        rows, cols = _sample_positions(m, K, 512, 20 + g)
        _check_sampled(dx[s0:s0 + m].cpu(), 2, da, db, Nn, rows, cols, f"expert {g} dgrad")
        # wgrad: MXFP8 columns over the expert's 128-padded tokens
        xp = np.zeros((mp, K), np.uint16); xp[:m] = xb[s0:s0 + m]
        dp = np.zeros((mp, Nn), np.uint16); dp[:m] = dyb[s0:s0 + m]
        wa = oracle.mxfp8_quantize_cols(dp) + (0.0,)
        wbb = oracle.mxfp8_quantize_cols(xp) + (0.0,)
        assert_codes_equal(dyc_c[:, p0:p0 + mp], wa[0], f"expert {g} dy_col codes")
        assert np.array_equal(dyc_s[:, p0 // 32:(p0 + mp) // 32], wa[1]), f"expert {g} dy_col scales"
        assert_codes_equal(xc_c[:, p0:p0 + mp], wbb[0], f"expert {g} x_col codes")
        assert np.array_equal(xc_s[:, p0 // 32:(p0 + mp) // 32], wbb[1]), f"expert {g} x_col scales"
        rows, cols = _sample_positions(Nn, K, 512, 30 + g)
        _check_sampled(dw[g].cpu(), 2, wa, wbb, mp, rows, cols, f"expert {g} wgrad")


def test_moe_grouped_nvfp4_backward_full_size():
    """The MoE workload with an NVFP4 backward ("MXFP8 fwd and NVFP4 bwd (or vice
    versa)"): dy grouped with SR in both directions and RHT on the columns, x
    columns with RHT, W columns; grouped NVFP4 dgrad and wgrad.  For a spread of
    experts the operands are bit-exact against the oracle at their padded
    positions (the stochastic-rounding index of a grouped element), and sampled
    outputs are within the GEMM tolerance."""
    sizes, x, w, dy = inputs.moe_grouped()
    G, Nn, K = w.shape
    sizes = [int(v) for v in sizes]
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    dyr, dyc = nvq.grouped_hybrid_quantize(dy.cuda(), sizes, nvq.NVFP4, nvq.NVFP4, rht_sign=sign, sr=sr)
    _, xc = nvq.grouped_hybrid_quantize(x.cuda(), sizes, nvq.NONE, nvq.NVFP4, rht_sign=sign)
    _, wc = nvq.grouped_hybrid_quantize(w.reshape(G * Nn, K).cuda(), [Nn] * G, nvq.NONE, nvq.NVFP4)
    dx = nvq.grouped_gemm_rows(dyr, wc, sizes, Nn, b_col_groups=True)
    dw = nvq.grouped_gemm_wgrad(dyc, xc, sizes)
    torch.cuda.synchronize()

    order = np.argsort(sizes)
    picks = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[len(order) // 2]), 9]))
    offs = np.concatenate([[0], np.cumsum(sizes)])
    poffs = np.concatenate([[0], np.cumsum([-(-m // 128) * 128 for m in sizes])])
    P = int(poffs[-1])
    xb, wb, dyb = bits(x), bits(w), bits(dy)
    dyr_c, dyc_c, xc_c, wc_c = qt_codes(dyr), qt_codes(dyc), qt_codes(xc), qt_codes(wc)
    dyr_s = oracle.scale_unswizzle(qt_scales(dyr), P, Nn // 16)
    dyc_s = oracle.scale_unswizzle(qt_scales(dyc), Nn, P // 16)
    xc_s = oracle.scale_unswizzle(qt_scales(xc), K, P // 16)
    wc_s = oracle.scale_unswizzle(qt_scales(wc), K, G * Nn // 16)
    for g in picks:
        m, s0, p0 = sizes[g], int(offs[g]), int(poffs[g])
        mp = -(-m // 128) * 128
        # W_g columns (contraction N), as dgrad's B operand
        wcc, wcs, wa = oracle.nvfp4_quantize_cols(wb[g])
        assert wc.amax[g].item() == np.float32(wa), f"expert {g} w_col amax"
        assert_codes_equal(wc_c[:, g * Nn // 2:(g + 1) * Nn // 2], wcc, f"expert {g} w_col codes")
        assert np.array_equal(wc_s[:, g * Nn // 16:(g + 1) * Nn // 16], wcs), f"expert {g} w_col scales"
        # dy_g rows (SR) at padded rows p0..
        dg = dyb[s0:s0 + m]
        A_r = oracle.amax(dg)
        assert dyr.amax[g].item() == np.float32(A_r), f"expert {g} dy_row amax"
        rc, rs = oracle.nvfp4_quantize_rows_at(dg, A_r, p0, sr=sr)
        assert_codes_equal(dyr_c[p0:p0 + m], rc, f"expert {g} dy_row codes")
        assert np.array_equal(dyr_s[p0:p0 + m], rs), f"expert {g} dy_row scales"
        # dy_g and x_g columns (RHT; SR for dy) over the zero-padded group
        dp = np.zeros((mp, Nn), np.uint16); dp[:m] = dg
        xp = np.zeros((mp, K), np.uint16); xp[:m] = xb[s0:s0 + m]
        A_dc, A_xc = oracle.amax_rht_col(dg, sign), oracle.amax_rht_col(xb[s0:s0 + m], sign)
        assert dyc.amax[g].item() == np.float32(A_dc), f"expert {g} dy_col amax"
        assert xc.amax[g].item() == np.float32(A_xc), f"expert {g} x_col amax"
        dcc, dcs = oracle.nvfp4_quantize_cols_at(dp, A_dc, p0, P, rht_sign=sign, sr=sr)
        xcc, xcs = oracle.nvfp4_quantize_cols_at(xp, A_xc, p0, P, rht_sign=sign)
        assert_codes_equal(dyc_c[:, p0 // 2:(p0 + mp) // 2], dcc, f"expert {g} dy_col codes")
        assert np.array_equal(dyc_s[:, p0 // 16:(p0 + mp) // 16], dcs), f"expert {g} dy_col scales"
        assert_codes_equal(xc_c[:, p0 // 2:(p0 + mp) // 2], xcc, f"expert {g} x_col codes")
        assert np.array_equal(xc_s[:, p0 // 16:(p0 + mp) // 16], xcs), f"expert {g} x_col scales"
        # sampled outputs from the oracle's own operands
        rows, cols = _sample_positions(m, K, 512, 30 + g)
        _check_sampled(dx[s0:s0 + m].cpu(), 1, (rc, rs, A_r), (wcc, wcs, wa), Nn, rows, cols, f"expert {g} dgrad")
        rows, cols = _sample_positions(Nn, K, 512, 40 + g)
        _check_sampled(dw[g].cpu(), 1, (dcc, dcs, A_dc), (xcc, xcs, A_xc), mp, rows, cols, f"expert {g} wgrad")
