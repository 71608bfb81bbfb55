"""Parity at the Qwen3-8B-shaped linear stack's shapes, on the stack's own
seeded inputs, in the launch configuration the benchmark's stack workload
uses ("Add an NVFP4 quantization converter", "What changed": the
qwen3_8b_nvfp4_mixed config; hidden 4096, 1024-wide k/v, MLP 12288, 2048 x 8
tokens).

One NVFP4 layer is composed as the benchmark composes it: q, k, v, gate and
up read the layer input h; o reads q's output and down reads up's output; the
backward quantizes each output gradient (stochastic rounding, Hadamard
transform on the columnwise copy) and runs dgrad and wgrad against the saved
operands.  Every quantized operand is compared with the oracle bit for bit
(codes, swizzled scales, amax); every GEMM output on sampled entries that the
oracle computes one by one from its own operands (relative Frobenius error
<= 1e-3, >= 99.9% within one bf16 ulp).

The o and down inputs: the oracle computes q's and up's outputs in full
(dequantized operands, fp64 product, one rounding to bf16), those outputs are
checked against the GPU's, and the oracle's outputs are then the o and down
inputs on both sides, so no input of the oracle comes from the GPU path."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

from gpu_util import (assert_codes_equal, assert_gemm_close, assert_scales_equal, bf16_from_bits, bits,
                      check_sampled_gemm, qt_codes, sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def _check_q(q, ref, what):
    c, s, A = ref
    assert q.amax.item() == np.float32(A), f"{what} amax {q.amax.item()} vs {A}"
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")


def _deq(t):
    c, s, A = t
    return oracle.nvfp4_dequant(c, s, oracle.nvfp4_g(A))


def test_qwen3_8b_nvfp4_layer_full_size():
    cfg = inputs.QWEN3_8B_STACK
    Tk, H, KV, F = cfg["tokens"], cfg["hidden"], cfg["kv_dim"], cfg["mlp"]
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    cc = nvq.colwise_cols
    al = nvq.alloc_qtensor

    # the stack's seeded inputs (drawn on the device, as the benchmark draws them)
    h = inputs.normal_bf16_on((Tk, H), 1.0, 1, "cuda")
    ws = dict(inputs.qwen3_layer_weights(0, device="cuda"))
    dys = {n: inputs.normal_bf16_on((Tk, n), 0.01, 2, "cuda") for n in (H, KV, F)}
    src = {"q": "h", "k": "h", "v": "h", "gate": "h", "up": "h", "o": "attn", "down": "mlp"}

    # ---------------- forward on the GPU, in the benchmark's order and calls
    act = {k: (al(nvq.NVFP4, Tk, d), al(nvq.NVFP4, d, cc(nvq.NVFP4, Tk))) for k, d in (("h", H), ("attn", H), ("mlp", F))}
    wq = {n: (al(nvq.NVFP4, W.shape[0], W.shape[1]), al(nvq.NVFP4, W.shape[1], cc(nvq.NVFP4, W.shape[0])))
          for n, W in ws.items()}
    y = {n: torch.empty(Tk, W.shape[0], dtype=torch.bfloat16, device="cuda") for n, W in ws.items()}
    nvq.nvfp4_quantize(h, 3, rht_sign=sign, out_row=act["h"][0], out_col=act["h"][1])
    for n in ("q", "k", "v", "gate", "up"):
        nvq.nvfp4_quantize(ws[n], 3, out_row=wq[n][0], out_col=wq[n][1])
        nvq.gemm_tn(act["h"][0], wq[n][0], out=y[n])
    torch.cuda.synchronize()

    # ---------------- oracle: layer input, weights, first five outputs
    hb = bits(h)
    ref_h = (oracle.nvfp4_quantize_rows(hb), oracle.nvfp4_quantize_cols(hb, rht_sign=sign))
    _check_q(act["h"][0], ref_h[0], "h row")
    _check_q(act["h"][1], ref_h[1], "h col (RHT)")
    ref_w = {}
    for n, W in ws.items():
        wb = bits(W)
        ref_w[n] = (oracle.nvfp4_quantize_rows(wb), oracle.nvfp4_quantize_cols(wb))
    for i, n in enumerate(("q", "k", "v", "gate", "up")):
        _check_q(wq[n][0], ref_w[n][0], f"W_{n} row")
        _check_q(wq[n][1], ref_w[n][1], f"W_{n} col")
        No = ws[n].shape[0]
        check_sampled_gemm(y[n], 1, ref_h[0], ref_w[n][0], H, *sample_positions(Tk, No, 2048, 40 + i, line=1024),
                           f"fwd {n}")

    # q's and up's outputs in full (the o and down inputs), from the oracle's own operands
    y_ref = {}
    for n in ("q", "up"):
        ref64 = oracle.gemm_tn_f64_blas(_deq(ref_h[0]), _deq(ref_w[n][0]))
        assert_gemm_close(y[n], ref64, f"fwd {n} (full)")
        y_ref[n] = bf16_from_bits(oracle.to_bf16_rne(ref64))
        del ref64

    # ---------------- o and down on the oracle's q / up outputs
    y_in = {"attn": y_ref["q"].cuda(), "mlp": y_ref["up"].cuda()}
    for n, a in (("o", "attn"), ("down", "mlp")):
        nvq.nvfp4_quantize(y_in[a], 3, rht_sign=sign, out_row=act[a][0], out_col=act[a][1])
        nvq.nvfp4_quantize(ws[n], 3, out_row=wq[n][0], out_col=wq[n][1])
        nvq.gemm_tn(act[a][0], wq[n][0], out=y[n])
    torch.cuda.synchronize()
    ref_a = {}
    for n, a in (("o", "attn"), ("down", "mlp")):
        ab = bits(y_ref["q" if a == "attn" else "up"])
        ref_a[a] = (oracle.nvfp4_quantize_rows(ab), oracle.nvfp4_quantize_cols(ab, rht_sign=sign))
        _check_q(act[a][0], ref_a[a][0], f"{a} row")
        _check_q(act[a][1], ref_a[a][1], f"{a} col (RHT)")
        _check_q(wq[n][0], ref_w[n][0], f"W_{n} row")
        _check_q(wq[n][1], ref_w[n][1], f"W_{n} col")
        Ki, No = ws[n].shape[1], ws[n].shape[0]
        check_sampled_gemm(y[n], 1, ref_a[a][0], ref_w[n][0], Ki, *sample_positions(Tk, No, 2048, 50, line=1024),
                           f"fwd {n}")
    ref_in = {"h": ref_h, **ref_a}

    # ---------------- backward (reverse order), as the benchmark runs it
    ref_dy = {}
    for i, n in enumerate(("down", "o", "up", "gate", "v", "k", "q")):
        No, Ki = ws[n].shape
        b = nvq.nvfp4_linear_bwd_quantize(dys[No], rht_sign=sign, sr=sr)
        dx = nvq.nvfp4_linear_dgrad(b["dy_row"], wq[n][1])
        dw = nvq.nvfp4_linear_wgrad(b["dy_col"], act[src[n]][1])
        torch.cuda.synchronize()
        if No not in ref_dy:
            db = bits(dys[No])
            ref_dy[No] = (oracle.nvfp4_quantize_rows(db, sr=sr), oracle.nvfp4_quantize_cols(db, rht_sign=sign, sr=sr))
        _check_q(b["dy_row"], ref_dy[No][0], f"dy[{No}] row (SR) for {n}")
        _check_q(b["dy_col"], ref_dy[No][1], f"dy[{No}] col (RHT, SR) for {n}")
        assert dx.shape == (Tk, Ki) and dw.shape == (No, Ki)
        check_sampled_gemm(dx, 1, ref_dy[No][0], ref_w[n][1], No, *sample_positions(Tk, Ki, 2048, 60 + i, line=1024),
                           f"dgrad {n}")
        check_sampled_gemm(dw, 1, ref_dy[No][1], ref_in[src[n]][1], Tk,
                           *sample_positions(No, Ki, 2048, 70 + i, line=1024), f"wgrad {n}")
