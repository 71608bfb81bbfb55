"""Row-scaled NVFP4 on the GPU against the oracle ("Hybrid quantization",
Description: the Composer-style grouped GEMM recipe, row-scaled NVFP4 forward
+ MXFP8 backward, with NVFP4Quantizer(row_scaled_nvfp4=True) as the grouped
linear's input quantizer): per-row amaxes, codes and swizzled scales bit for
bit; GEMMs with a row-scaled A (alpha per output row) within the GEMM
tolerance, on both GEMM kernels and on the grouped GEMM; the grouped linear
forward with a row-scaled input at the MoE workload's full size."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import (assert_codes_equal, assert_gemm_close, assert_scales_equal, bits, check_mxfp8_col,
                      check_sampled_gemm, qt_codes, sample_positions)

pytestmark = pytest.mark.gpu
RS = nvq.NVFP4_ROWSCALED


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _check_rows(q, x, what="row-scaled rows"):
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(bits(x))
    got_a = q.amax[: a.size].cpu().numpy()
    assert np.array_equal(got_a, a), f"{what}: per-row amax"
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s, a


@pytest.mark.parametrize("M,K", [(256, 512), (300, 96), (40, 64), (129, 272)])
@pytest.mark.parametrize("col_fmt", [nvq.NONE, nvq.MXFP8])
def test_row_scaled_quantize(M, K, col_fmt):
    x = inputs.student_t3_outliers(M, K)
    row, col = nvq.hybrid_quantize(x.cuda(), RS, col_fmt)
    torch.cuda.synchronize()
    _check_rows(row, x)
    if col_fmt == nvq.MXFP8:
        check_mxfp8_col(col, x)


@pytest.mark.parametrize("N", [256, 384])  # CTA-pair kernel and single-CTA kernel
def test_gemm_with_row_scaled_a(N):
    M, K = 384, 512
    x = inputs.student_t3_outliers(M, K)
    x[5] = 0  # a zero row: alpha 0
    w = inputs.normal_bf16((N, K), 0.02, torch.Generator().manual_seed(N))
    xr, _ = nvq.hybrid_quantize(x.cuda(), RS, nvq.NONE)
    wr, _ = nvq.nvfp4_quantize(w.cuda(), nvq.DIR_ROW)
    bias = inputs.normal_bf16((1, N), 1.0, torch.Generator().manual_seed(3)).reshape(N)
    y32 = nvq.gemm_tn(xr, wr, bias=bias.cuda(), out_dtype=torch.float32)
    y16 = nvq.gemm_tn(xr, wr, bias=bias.cuda())
    torch.cuda.synchronize()
    c, s, a = _check_rows(xr, x)
    wc, ws, wa = oracle.nvfp4_quantize_rows(bits(w))
    ref = oracle.gemm_tn_f64(oracle.nvfp4_dequant_rowscaled(c, s, a), oracle.nvfp4_dequant(wc, ws, oracle.nvfp4_g(wa)),
                             bias=bias.float().numpy())
    assert_gemm_close(y32, ref, f"row-scaled fp32 N={N}")
    assert_gemm_close(y16, ref, f"row-scaled bf16 N={N}")


def _padded_rowscaled(x, sizes):
    """Oracle row-scaled rows placed in the grouped (128-row padded) layout."""
    c, s, a = oracle.nvfp4_quantize_rows_rowscaled(bits(x))
    P = sum(-(-m // 128) * 128 for m in sizes)
    K = bits(x).shape[1]
    cp = np.zeros((P, K // 2), np.uint8)
    sp = np.zeros((P, K // 16), np.uint8)
    ap = np.zeros(P, np.float32)
    src = dst = 0
    for m in sizes:
        cp[dst:dst + m], sp[dst:dst + m], ap[dst:dst + m] = c[src:src + m], s[src:src + m], a[src:src + m]
        src += m
        dst += -(-m // 128) * 128
    return cp, sp, ap


def test_grouped_row_scaled_quantize_and_gemm():
    sizes = [5, 0, 130, 1, 256, 77]
    G, K, N = len(sizes), 256, 256
    x = inputs.normal_bf16((sum(sizes), K), 1.0, torch.Generator().manual_seed(31))
    w = inputs.normal_bf16((G * N, K), 0.02, torch.Generator().manual_seed(32))
    xr, xc = nvq.grouped_hybrid_quantize(x.cuda(), sizes, RS, nvq.MXFP8)
    wr, _ = nvq.grouped_hybrid_quantize(w.cuda(), [N] * G, nvq.NVFP4, nvq.NONE)
    y = nvq.grouped_gemm_rows(xr, wr, sizes, N, b_col_groups=False)
    torch.cuda.synchronize()
    cp, sp, ap = _padded_rowscaled(x, sizes)
    assert np.array_equal(xr.amax.cpu().numpy(), ap)
    assert_codes_equal(qt_codes(xr), cp, "grouped row-scaled codes")
    assert_scales_equal(xr, sp, "grouped row-scaled scales")
    wb = bits(w)
    off = pofs = 0
    for g, m in enumerate(sizes):
        if m:
            wq = oracle.nvfp4_quantize_rows(wb[g * N:(g + 1) * N])
            ref = oracle.gemm_tn_f64(oracle.nvfp4_dequant_rowscaled(cp[pofs:pofs + m], sp[pofs:pofs + m], ap[pofs:pofs + m]),
                                     oracle.nvfp4_dequant(wq[0], wq[1], oracle.nvfp4_g(wq[2])))
            assert_gemm_close(y[off:off + m], ref, f"expert {g}")
        off += m
        pofs += -(-m // 128) * 128


def test_grouped_linear_row_scaled_input_moe_full_size():
    """The MoE workload (64 experts 4096 -> 1536, 65536 Zipf(1.1) tokens) with
    the Composer-style input: row-scaled NVFP4 forward; sampled outputs of a
    spread of experts against the oracle, every expert's input rows bit-exact."""
    sizes, x, w, _ = inputs.moe_grouped()
    G, Nn, K = w.shape
    sizes = [int(v) for v in sizes]
    y, bufs = nvq.grouped_linear_fwd(x.cuda(), w.reshape(G * Nn, K).cuda(), sizes, row_scaled_x=True)
    torch.cuda.synchronize()
    xr = bufs["x_row"]
    assert xr.fmt == RS
    cp, sp, ap = _padded_rowscaled(x, sizes)
    assert np.array_equal(xr.amax.cpu().numpy(), ap)
    assert_codes_equal(qt_codes(xr), cp, "MoE row-scaled x codes")
    assert_scales_equal(xr, sp, "MoE row-scaled x scales")
    order = np.argsort(sizes)
    picks = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[len(order) // 2]), 7]))
    offs = np.concatenate([[0], np.cumsum(sizes)])
    poffs = np.concatenate([[0], np.cumsum([-(-m // 128) * 128 for m in sizes])])
    wb = bits(w)
    for g in picks:
        m, s0, p0 = sizes[g], int(offs[g]), int(poffs[g])
        if m == 0:
            continue
        wq = oracle.nvfp4_quantize_rows(wb[g])
        rows, cols = sample_positions(m, Nn, 512, 90 + g)
        ref = oracle.gemm_tn_sampled_rowscaled(cp[p0:p0 + m], sp[p0:p0 + m], ap[p0:p0 + m], wq[0], wq[1], wq[2], K,
                                               rows, cols)
        got = y[s0:s0 + m][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
        refb = torch.from_numpy(oracle.to_bf16_rne(ref).view(np.int16)).view(torch.bfloat16).float().numpy()
        rel = np.linalg.norm(got - refb) / np.linalg.norm(refb)
        assert rel <= 1e-3, f"expert {g}: sampled relative Frobenius error {rel:.3e}"
