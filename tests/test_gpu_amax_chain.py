"""The tensor amax produced upstream: a GEMM whose epilogue also writes the
amaxes of its output (plain, and over the Hadamard-transformed 16-row column
blocks), and quantization that takes a given amax instead of measuring it
("Add an NVFP4 quantization converter", "What changed": every NVFP4 input
carries an FP32 per-tensor scale; the amax that sets it can come from the
operation that produced the tensor).

* On operands whose products are exact, the GPU output equals the oracle's
  bit for bit, so the epilogue amaxes must equal the oracle's amaxes of the
  oracle's own output exactly.
* Quantization with the given (oracle) amax is bit-exact against the oracle.
* In a chain of layers, the next layer's quantization with the amaxes the
  previous GEMM wrote equals its quantization with measured amaxes, byte for
  byte, and the written amaxes equal the measured ones."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import bf16_from_bits, bits, check_nvfp4_col, check_nvfp4_row

pytestmark = pytest.mark.gpu
SIGN = inputs.rht_sign_vector()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _exact_operand(rows, K, rng, special_block):
    """E2M1 grid values times powers of two per 16-block (block max 6 s), one
    value 2688 in a reserved block so the tensor amax is 2688 (g = 1)."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    x = np.zeros((rows, K))
    for i in range(rows):
        for j in range(2, K // 16):
            s = 2.0 ** rng.integers(-2, 2)
            c = rng.choice(grid, 16) * rng.choice([-1, 1], 16)
            c[rng.integers(16)] = 6.0
            x[i, 16 * j:16 * j + 16] = c * s
    x[0, 16 * special_block] = 2688.0
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("N", [256, 384])  # CTA-pair kernel and single-CTA kernel
@pytest.mark.parametrize("c_fp32", [False, True])
def test_epilogue_amax_equals_oracle_on_exact_products(N, c_fp32):
    rng = np.random.default_rng(5)
    a = _exact_operand(256, 512, rng, special_block=0)
    b = _exact_operand(N, 512, rng, special_block=1)
    ar, _ = nvq.nvfp4_quantize(a.cuda(), nvq.DIR_ROW)
    br, _ = nvq.nvfp4_quantize(b.cuda(), nvq.DIR_ROW)
    am = torch.full((1,), -1.0, device="cuda")
    ar_ = torch.full((1,), -1.0, device="cuda")
    y = nvq.gemm_tn(ar, br, out_dtype=torch.float32 if c_fp32 else torch.bfloat16, rht_sign=SIGN, amax_out=am,
                    amax_rht_out=ar_)
    torch.cuda.synchronize()
    ac, asc, Aa = oracle.nvfp4_quantize_rows(bits(a))
    bc, bsc, Ab = oracle.nvfp4_quantize_rows(bits(b))
    ref = oracle.gemm_tn_f64(oracle.nvfp4_dequant(ac, asc, oracle.nvfp4_g(Aa)),
                             oracle.nvfp4_dequant(bc, bsc, oracle.nvfp4_g(Ab)))
    if c_fp32:
        ref32 = ref.astype(np.float32)
        assert np.array_equal(ref32.astype(np.float64), ref)  # the products are exact in fp32
        assert np.array_equal(y.cpu().numpy(), ref32)
        # the oracle amaxes of an fp32 tensor, through its exact bf16 rounding
        # would lose bits: take them from the fp32 values with the oracle's
        # butterfly on each 16-row column block
        want = float(np.max(np.abs(ref32)))
        u = ref32.reshape(-1, 16, N).transpose(0, 2, 1).reshape(-1, 16)
        want_rht = max(float(np.max(np.abs(oracle.rht16(row, SIGN)))) for row in u)
    else:
        yb = oracle.to_bf16_rne(ref)
        assert np.array_equal(bits(y), yb)
        want = oracle.amax(yb)
        want_rht = oracle.amax_rht_col(yb, SIGN)
    assert am.item() == np.float32(want)
    assert ar_.item() == np.float32(want_rht)


def test_quantize_with_given_amax_is_oracle_exact():
    x = inputs.normal_bf16((384, 512), 1.0, torch.Generator().manual_seed(17))
    xb = bits(x)
    A, A_rht = oracle.amax(xb), oracle.amax_rht_col(xb, SIGN)
    row = nvq.alloc_qtensor(nvq.NVFP4, 384, 512)
    col = nvq.alloc_qtensor(nvq.NVFP4, 512, nvq.colwise_cols(nvq.NVFP4, 384))
    row.amax.fill_(float(A))
    col.amax.fill_(float(A_rht))
    nvq.nvfp4_quantize(x.cuda(), 3, rht_sign=SIGN, sr=(77, 1), out_row=row, out_col=col, amax_given=True)
    torch.cuda.synchronize()
    check_nvfp4_row(row, x, sr=(77, 1))
    check_nvfp4_col(col, x, rht=SIGN, sr=(77, 1))


def test_amax_given_from_the_previous_layer_equals_measured():
    """Two NVFP4 linears in a row (x -> y1 -> y2) and a dgrad whose dx is the
    next output gradient: the amaxes a GEMM writes equal the ones the amax
    pass measures on its output, and the downstream quantization with the
    given amaxes equals the one that measures them."""
    M, K, N1, N2 = 512, 768, 1024, 256
    g = torch.Generator().manual_seed(23)
    x = inputs.normal_bf16((M, K), 1.0, g).cuda()
    w1 = inputs.normal_bf16((N1, K), 0.02, g).cuda()
    w2 = inputs.normal_bf16((N2, N1), 0.02, g).cuda()
    dy2 = inputs.normal_bf16((M, N2), 0.01, g).cuda()
    sr = (inputs.SR_SEED, 0)
    # layer 1 writes y1's amaxes straight into layer 2's input buffers
    l2 = dict(x_row=nvq.alloc_qtensor(nvq.NVFP4, M, N1), w_row=nvq.alloc_qtensor(nvq.NVFP4, N2, N1),
              x_col=nvq.alloc_qtensor(nvq.NVFP4, N1, M), w_col=nvq.alloc_qtensor(nvq.NVFP4, N1, N2))
    y1, l1 = nvq.nvfp4_linear_fwd(x, w1, rht_sign=SIGN, y_amax=l2["x_row"].amax, y_amax_rht=l2["x_col"].amax)
    y2, l2 = nvq.nvfp4_linear_fwd(y1, w2, rht_sign=SIGN, bufs=l2, amax_given=True)
    # the same layer 2 with measured amaxes
    y2m, l2m = nvq.nvfp4_linear_fwd(y1, w2, rht_sign=SIGN)
    a_plain, a_rht = nvq.amax(y1, rht_sign=SIGN)
    # backward of layer 2: its dgrad writes dx2's amaxes into layer 1's dy buffers
    b2 = nvq.nvfp4_linear_bwd_quantize(dy2, rht_sign=SIGN, sr=sr)
    b1 = dict(dy_row=nvq.alloc_qtensor(nvq.NVFP4, M, N1), dy_col=nvq.alloc_qtensor(nvq.NVFP4, N1, M))
    dx2 = nvq.nvfp4_linear_dgrad(b2["dy_row"], l2["w_col"], rht_sign=SIGN, dx_amax=b1["dy_row"].amax,
                                 dx_amax_rht=b1["dy_col"].amax)
    b1 = nvq.nvfp4_linear_bwd_quantize(dx2, rht_sign=SIGN, sr=sr, bufs=b1, amax_given=True)
    b1m = nvq.nvfp4_linear_bwd_quantize(dx2, rht_sign=SIGN, sr=sr)
    torch.cuda.synchronize()
    assert l2["x_row"].amax.item() == a_plain.item() and l2["x_col"].amax.item() == a_rht.item()
    for k in ("x_row", "x_col"):
        assert torch.equal(l2[k].data, l2m[k].data) and torch.equal(l2[k].scale, l2m[k].scale), k
        assert torch.equal(l2[k].amax, l2m[k].amax), k
    assert torch.equal(y2, y2m)
    for k in ("dy_row", "dy_col"):
        assert torch.equal(b1[k].data, b1m[k].data) and torch.equal(b1[k].scale, b1m[k].scale), k
        assert torch.equal(b1[k].amax, b1m[k].amax), k
