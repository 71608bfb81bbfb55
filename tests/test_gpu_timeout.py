"""Failure detection without a GPU fault: every pipeline wait in the GEMM is
bounded.  With the NVQ_DEBUG_DROP_TMA test hook the kernel's first stage is
armed but never filled; the waits run out (about 2 s each), the kernel records
NVQ_ERR_TIMEOUT in the device status word, releases its TMEM and returns, and
the context stays usable: the next GEMM is correct."""
import os

import pytest
import torch

import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import __graft_entry__
    __graft_entry__.build()
    x, w = inputs.single_linear()
    xr, _ = nvq.nvfp4_quantize(x.cuda(), nvq.DIR_ROW)
    wr, _ = nvq.nvfp4_quantize(w.cuda(), nvq.DIR_ROW)
    good = nvq.gemm_tn(xr, wr)
    torch.cuda.synchronize()
    assert nvq.device_status() == 0
    os.environ["NVQ_DEBUG_DROP_TMA"] = "1"
    try:
        nvq.gemm_tn(xr, wr)
        assert nvq.device_status() == 7  # NVQ_ERR_TIMEOUT, status word cleared by the read
    finally:
        del os.environ["NVQ_DEBUG_DROP_TMA"]
    again = nvq.gemm_tn(xr, wr)
    torch.cuda.synchronize()
    assert nvq.device_status() == 0
    assert torch.equal(again, good)
