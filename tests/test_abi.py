"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/nvq.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import build as nvq_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nvq.h")


@pytest.fixture(scope="module")
def lib():
    nvq_build.build()
    return nvq.load()


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(nvq_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_binding_surface():
    assert set(_declared()) == set(nvq.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_no_unexpected_cuda_symbols_leak(lib):
    # hidden visibility: internal kernels / helpers are not part of the ABI
    assert not hasattr(lib, "_ZN3nvq14launch_quantizeERKNS_9QuantArgsEiibblP11CUstream_st")


def test_status_strings(lib):
    for code in range(9):
        assert lib.nvq_status_string(code)
    assert lib.nvq_version().startswith(b"nvq")


def test_query_sizes():
    assert nvq.query_sizes(nvq.NVFP4, 256, 512) == (256 * 256, 256 * 32)
    assert nvq.query_sizes(nvq.IDENTITY, 40, 48) == (40 * 48 * 2, 0)
    assert nvq.colwise_cols(nvq.IDENTITY, 40) == 48
    assert nvq.query_sizes(nvq.MXFP8, 200, 96) == (200 * 96, 256 * 4)
    assert nvq.colwise_cols(nvq.NVFP4, 40) == 48
    assert nvq.colwise_cols(nvq.MXFP8, 48) == 64
    with pytest.raises(nvq.NvqError):
        nvq.query_sizes(nvq.NVFP4, 16, 24)  # cols not a multiple of 16
    with pytest.raises(nvq.NvqError):
        nvq.query_sizes(7, 16, 32)


def test_grouped_padded_rows():
    assert nvq.grouped_padded_rows([0, 1, 128, 129]) == 0 + 128 + 128 + 256
    assert nvq.load().nvq_grouped_padded_rows(None, 3) == -1


def _qt(fmt, rows, cols, data=16, scale=16, amax=16):
    return nvq._QT(fmt, data, scale, amax, rows, cols)


def test_host_validation_before_any_launch(lib):
    """Argument errors come back as status codes without a device."""
    QTP = ctypes.byref
    r = _qt(nvq.NVFP4, 128, 256)
    c = _qt(nvq.NVFP4, 256, 128)
    # NULL input
    assert lib.nvq_nvfp4_quantize(None, 128, 256, 256, 3, None, None, QTP(r), QTP(c), None) == 1
    # ld < K
    assert lib.nvq_nvfp4_quantize(16, 128, 256, 128, 3, None, None, QTP(r), QTP(c), None) == 2
    # misaligned input
    assert lib.nvq_nvfp4_quantize(18, 128, 256, 256, 3, None, None, QTP(r), QTP(c), None) == 3
    # K not a multiple of 16
    assert lib.nvq_nvfp4_quantize(16, 128, 24, 24, 1, None, None, QTP(_qt(1, 128, 24)), None, None) == 2
    # output shape mismatch
    assert lib.nvq_nvfp4_quantize(16, 128, 256, 256, 1, None, None, QTP(_qt(1, 64, 256)), None, None) == 2
    # NVFP4 output without amax storage
    assert lib.nvq_nvfp4_quantize(16, 128, 256, 256, 1, None, None, QTP(_qt(1, 128, 256, amax=None)), None, None) == 1
    # MXFP8 rowwise needs K % 32
    assert lib.nvq_mxfp8_quantize(16, 128, 48, 48, 1, QTP(_qt(2, 128, 48)), None, None) == 2
    # hybrid: columnwise_source must be original (0) or rowwise_dequantized (1), and the
    # rowwise-dequantized source needs a quantized rowwise direction
    assert lib.nvq_hybrid_quantize(16, 128, 256, 256, 1, 2, 2, None, None, QTP(r), QTP(c), None) == 5
    assert lib.nvq_hybrid_quantize(16, 128, 256, 256, 0, 2, 1, None, None, None, QTP(c), None) == 5
    assert lib.nvq_hybrid_quantize(16, 128, 256, 256, 3, 2, 1, None, None, QTP(_qt(3, 128, 256)), QTP(c), None) == 5
    # identity is a quantize direction only: no grouped identity, no identity GEMM
    rows2 = (ctypes.c_int64 * 2)(3, 5)
    assert lib.nvq_grouped_hybrid_quantize(16, 256, 256, rows2, 2, 3, 2, QTP(_qt(3, 256, 256)), QTP(c), None, None,
                                           None) == 5
    assert lib.nvq_gemm_tn(QTP(_qt(3, 128, 256)), QTP(_qt(3, 128, 256)), None, 16, 128, 0, None) == 5
    # bad RHT sign vector
    bad = nvq._RHT((ctypes.c_int8 * 16)(*([1] * 15 + [0])))
    assert lib.nvq_nvfp4_quantize(16, 128, 256, 256, 3, QTP(bad), None, QTP(r), QTP(c), None) == 2
    # GEMM: rows not a multiple of 128, mismatched formats, mismatched K
    A = _qt(1, 100, 256)
    B = _qt(1, 128, 256)
    assert lib.nvq_gemm_tn(QTP(A), QTP(B), None, 16, 128, 0, None) == 2
    assert lib.nvq_gemm_tn(QTP(_qt(1, 128, 256)), QTP(_qt(2, 128, 256)), None, 16, 128, 0, None) == 5
    assert lib.nvq_gemm_tn(QTP(_qt(1, 128, 256)), QTP(_qt(1, 128, 384)), None, 16, 128, 0, None) == 2
    assert lib.nvq_gemm_tn(QTP(_qt(1, 128, 256)), QTP(_qt(1, 128, 256)), None, None, 128, 0, None) in (1, 6)
    # linear entry points: dims must be multiples of 128
    assert lib.nvq_nvfp4_linear_fwd(16, 16, None, 100, 128, 128, None, 16, QTP(r), QTP(r), None, None, None) == 2
    # grouped: SR / RHT validated like the ungrouped call (a sign entry other
    # than +-1 is a shape error), too many groups rejected
    rows = (ctypes.c_int64 * 2)(3, 5)
    bad_sign = nvq._RHT((ctypes.c_int8 * 16)(*([1] * 15 + [0])))
    assert lib.nvq_grouped_hybrid_quantize(16, 256, 256, rows, 2, 1, 1, QTP(_qt(1, 256, 256)),
                                           QTP(_qt(1, 256, 256)), ctypes.byref(bad_sign), None, None) == 2
    many = (ctypes.c_int64 * 300)(*([1] * 300))
    assert lib.nvq_grouped_hybrid_quantize(16, 256, 256, many, 300, 1, 2, QTP(r), QTP(c), None, None, None) == 2
