"""GPU block-scaled GEMMs (tcgen05) vs the oracle's fp64 product of its own
dequantized operands.

Tolerance: the fp32 output is within relative Frobenius error 1e-3 of the
fp64 oracle; the bf16 output is within 1e-3 of the oracle rounded once to
bf16 with >= 99.9% of elements within one bf16 ulp (bf16 output rounding
alone is ~1.5e-3 relative, so a bf16-vs-fp64 bound of 1e-3 could never hold).
Operands whose products and partial sums are exact in fp32 must give a
bit-exact fp32 output.

Pages: "Add an NVFP4 quantization converter" (NVFP4 linear, Table 1 path;
GEMM dims multiples of 128) and "Hybrid quantization" (MXFP8 GEMM)."""
import os

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import assert_gemm_close, bits, check_nvfp4_col, check_nvfp4_row

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


def _nv_ref(a, b, sr_a=None, bias=None):
    ac, asc, Aa = oracle.nvfp4_quantize_rows(bits(a), sr=sr_a)
    bc, bsc, Ab = oracle.nvfp4_quantize_rows(bits(b))
    return oracle.gemm_tn_f64(oracle.nvfp4_dequant(ac, asc, oracle.nvfp4_g(Aa)),
                              oracle.nvfp4_dequant(bc, bsc, oracle.nvfp4_g(Ab)), bias=bias)


def _mx_ref(a, b, bias=None):
    ac, asc = oracle.mxfp8_quantize_rows(bits(a))
    bc, bsc = oracle.mxfp8_quantize_rows(bits(b))
    return oracle.gemm_tn_f64(oracle.mxfp8_dequant(ac, asc), oracle.mxfp8_dequant(bc, bsc), bias=bias)


def test_single_linear_forward_workload():
    """x, W bf16[256,512] ~ N(0,1) seed 0, RTN rowwise NVFP4, y = x W^T bf16[256,256]."""
    x, w = inputs.single_linear()
    xr, _ = nvq.nvfp4_quantize(x.cuda(), nvq.DIR_ROW)
    wr, _ = nvq.nvfp4_quantize(w.cuda(), nvq.DIR_ROW)
    y = nvq.gemm_tn(xr, wr)
    y32 = nvq.gemm_tn(xr, wr, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = _nv_ref(x, w)
    assert_gemm_close(y32, ref, "single linear fp32")
    assert_gemm_close(y, ref, "single linear bf16")


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (384, 256, 384), (256, 384, 640), (512, 128, 1024)])
def test_multi_tile_and_k_tails(fmt, M, N, K):
    a = _randn(M, K, seed=M + 1)
    b = _randn(N, K, seed=N + 2, std=0.02)
    bias = _randn(1, N, seed=3).reshape(N)
    if fmt == 1:
        ar, _ = nvq.nvfp4_quantize(a.cuda(), nvq.DIR_ROW)
        br, _ = nvq.nvfp4_quantize(b.cuda(), nvq.DIR_ROW)
        ref = _nv_ref(a, b, bias=bias.float().numpy())
    else:
        ar, _ = nvq.mxfp8_quantize(a.cuda(), nvq.DIR_ROW)
        br, _ = nvq.mxfp8_quantize(b.cuda(), nvq.DIR_ROW)
        ref = _mx_ref(a, b, bias=bias.float().numpy())
    y32 = nvq.gemm_tn(ar, br, bias=bias.cuda(), out_dtype=torch.float32)
    y16 = nvq.gemm_tn(ar, br, bias=bias.cuda())
    torch.cuda.synchronize()
    assert_gemm_close(y32, ref, f"fmt{fmt} {M}x{N}x{K} fp32")
    assert_gemm_close(y16, ref, f"fmt{fmt} {M}x{N}x{K} bf16")


@pytest.mark.parametrize("fmt,K", [(1, 1152), (2, 896)])
def test_more_tiles_than_sm_pairs(fmt, K):
    """2048 x 2560 output: 80 CTA-pair tiles for at most 76 resident pairs on
    GB300, so some pairs run a second tile and carry the stage ring (slot,
    phase, descriptors, TMEM scale columns) across the tile boundary.  K = 1152
    (NVFP4) is 4.5 ring stages (a ragged last stage of 2 MMAs); K = 896 (MXFP8)
    is 7 stages, so the ring wraps inside each tile."""
    M, N = 2048, 2560
    if os.environ.get("NVQ_GEMM_PAIR") != "0":
        assert nvq.gemm_pair_available(), "output width 2560 should run on the CTA-pair kernel"
    a = _randn(M, K, seed=31)
    b = _randn(N, K, seed=32, std=0.05)
    if fmt == 1:
        ar, _ = nvq.nvfp4_quantize(a.cuda(), nvq.DIR_ROW)
        br, _ = nvq.nvfp4_quantize(b.cuda(), nvq.DIR_ROW)
        ref = _nv_ref(a, b)
    else:
        ar, _ = nvq.mxfp8_quantize(a.cuda(), nvq.DIR_ROW)
        br, _ = nvq.mxfp8_quantize(b.cuda(), nvq.DIR_ROW)
        ref = _mx_ref(a, b)
    y32 = nvq.gemm_tn(ar, br, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_gemm_close(y32, ref, f"fmt{fmt} {M}x{N}x{K} fp32")


def _exact_nvfp4_operand(rows, K, rng, special_block):
    """Blocks of E2M1 grid values c * s (s a power of two, block max 6 s); one
    block holds 2688 = 6 * 448 so the tensor amax is 2688 and g = A/2688 = 1."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    x = np.zeros((rows, K))
    for i in range(rows):
        for j in range(K // 16):
            if j in (0, 1):
                continue  # blocks 0 and 1 are reserved (see below)
            s = 2.0 ** rng.integers(-2, 2)
            c = rng.choice(grid, 16) * rng.choice([-1, 1], 16)
            c[rng.integers(16)] = 6.0
            x[i, 16 * j:16 * j + 16] = c * s
    x[0, 16 * special_block] = 2688.0  # only this operand's reserved block is nonzero
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def test_nvfp4_bit_exact_on_representable_operands():
    rng = np.random.default_rng(1)
    a = _exact_nvfp4_operand(256, 512, rng, special_block=0)
    b = _exact_nvfp4_operand(128, 512, rng, special_block=1)  # cross terms of blocks 0/1 vanish
    ar, _ = nvq.nvfp4_quantize(a.cuda(), nvq.DIR_ROW)
    br, _ = nvq.nvfp4_quantize(b.cuda(), nvq.DIR_ROW)
    y = nvq.gemm_tn(ar, br, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ar.amax.item() == 2688.0 and br.amax.item() == 2688.0
    ref = _nv_ref(a, b)
    exact = a.double().numpy() @ b.double().numpy().T  # quantization is exact here
    assert np.array_equal(ref, exact)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


def test_mxfp8_bit_exact_on_representable_operands():
    rng = np.random.default_rng(2)

    def operand(rows, K):
        x = np.zeros((rows, K))
        for i in range(rows):
            for j in range(K // 32):
                e = int(rng.integers(-4, 1))
                c = rng.choice([0, 256, 320, 384, 448], 32) * rng.choice([-1, 1], 32)
                c[rng.integers(32)] = 448
                x[i, 32 * j:32 * j + 32] = c * 2.0 ** e
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)

    a, b = operand(128, 512), operand(256, 512)
    ar, _ = nvq.mxfp8_quantize(a.cuda(), nvq.DIR_ROW)
    br, _ = nvq.mxfp8_quantize(b.cuda(), nvq.DIR_ROW)
    y = nvq.gemm_tn(ar, br, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = _mx_ref(a, b)
    assert np.array_equal(ref, a.double().numpy() @ b.double().numpy().T)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


def test_zero_amax_operand_gives_bias_only():
    a = torch.zeros(128, 256, dtype=torch.bfloat16)
    b = _randn(128, 256, seed=4)
    bias = _randn(1, 128, seed=5).reshape(128)
    ar, _ = nvq.nvfp4_quantize(a.cuda(), nvq.DIR_ROW)
    br, _ = nvq.nvfp4_quantize(b.cuda(), nvq.DIR_ROW)
    y = nvq.gemm_tn(ar, br, bias=bias.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), bias.float().expand(128, 128))


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (512, 384, 256)])
def test_linear_fwd_dgrad_wgrad(M, N, K):
    """NVFP4Linear forward + backward: RHT on the wgrad operands (shared sign
    vector), SR on dy in both directions, x and W round-to-nearest."""
    x = _randn(M, K, seed=10)
    w = _randn(N, K, seed=11, std=0.02)
    dy = _randn(M, N, seed=12, std=0.01)
    sr = (inputs.SR_SEED, 0)
    y, saved = nvq.nvfp4_linear_fwd(x.cuda(), w.cuda(), rht_sign=SIGN)
    bw = nvq.nvfp4_linear_bwd_quantize(dy.cuda(), rht_sign=SIGN, sr=sr)
    dx = nvq.nvfp4_linear_dgrad(bw["dy_row"], saved["w_col"])
    dw = nvq.nvfp4_linear_wgrad(bw["dy_col"], saved["x_col"])
    torch.cuda.synchronize()
    # every quantized operand bit-exact
    xr = check_nvfp4_row(saved["x_row"], x)
    wr = check_nvfp4_row(saved["w_row"], w)
    xc = check_nvfp4_col(saved["x_col"], x, rht=SIGN)
    wc = check_nvfp4_col(saved["w_col"], w)
    dr = check_nvfp4_row(bw["dy_row"], dy, sr=sr)
    dc = check_nvfp4_col(bw["dy_col"], dy, rht=SIGN, sr=sr)

    def deq(t):
        c, s, A = t
        return oracle.nvfp4_dequant(c, s, oracle.nvfp4_g(A))

    assert_gemm_close(y, oracle.gemm_tn_f64(deq(xr), deq(wr)), "fwd")
    assert_gemm_close(dx, oracle.gemm_tn_f64(deq(dr), deq(wc)), "dgrad")
    assert_gemm_close(dw, oracle.gemm_tn_f64(deq(dc), deq(xc)), "wgrad")
    # the Hadamard transforms cancel: wgrad approximates the plain dy^T x
    plain = bits(dy).astype(np.uint32) << 16
    dyf = plain.view(np.float32).astype(np.float64)
    xf = (bits(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rel = np.linalg.norm(dw.float().cpu().numpy() - dyf.T @ xf) / np.linalg.norm(dyf.T @ xf)
    assert rel < 0.25


@pytest.mark.parametrize("col_off", [128, 8])
def test_strided_output_matches_contiguous(col_off):
    """C written into a column slice of a wider tensor (ldc > N, base offset
    col_off elements: 256 B or 16 B) equals the contiguous result bit for bit,
    and nothing outside the slice is touched (both output paths: the CTA-pair
    kernel's TMA tensor stores and, under NVQ_GEMM_PAIR=0, the single-CTA
    kernel's 32-byte or 16-byte register stores)."""
    M, N, K = 384, 512, 512
    x = _randn(M, K, seed=21)
    w = _randn(N, K, seed=22, std=0.05)
    xr, _ = nvq.nvfp4_quantize(x.cuda(), nvq.DIR_ROW)
    wr, _ = nvq.nvfp4_quantize(w.cuda(), nvq.DIR_ROW)
    ref = nvq.gemm_tn(xr, wr)
    big = torch.full((M, N + 384), 7.0, dtype=torch.bfloat16, device="cuda")
    view = big[:, col_off:col_off + N]
    nvq.gemm_tn(xr, wr, out=view)
    torch.cuda.synchronize()
    assert view.stride(0) == N + 384
    assert torch.equal(view, ref)
    outside = torch.cat([big[:, :col_off], big[:, col_off + N:]], dim=1)
    assert torch.all(outside == 7.0)
