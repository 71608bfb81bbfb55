"""The grouped-linear entry points ("Hybrid quantization", Description: NVFP4
forward, MXFP8 backward for a grouped MoE linear) equal the composition of the
grouped quantize / GEMM calls they are built from, bit for bit, on a ragged
group table with an empty expert; the empty expert's weight gradient is zero.
The grouped calls themselves are checked against the oracle in
test_gpu_grouped.py."""
import pytest
import torch

import mxfp8_block_scaled_bf16_gb300 as nvq
from mxfp8_block_scaled_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert nvq.device_status() == 0


def test_grouped_linear_equals_its_composition():
    sizes = [130, 0, 257, 64]
    G, N, K = len(sizes), 256, 384
    T = sum(sizes)
    g = torch.Generator().manual_seed(11)
    x = inputs.normal_bf16((T, K), 1.0, g).cuda()
    w = inputs.normal_bf16((G, N, K), 0.02, g).cuda()
    dy = inputs.normal_bf16((T, N), 0.01, g).cuda()

    y, fb = nvq.grouped_linear_fwd(x, w, sizes)
    bb = nvq.grouped_linear_bwd_quantize(dy, sizes)
    dx = nvq.grouped_linear_dgrad(bb["dy_row"], fb["w_col"], sizes)
    dw = nvq.grouped_linear_wgrad(bb["dy_col"], fb["x_col"], sizes)

    w2 = w.reshape(G * N, K)
    xr, xc = nvq.grouped_hybrid_quantize(x, sizes, nvq.NVFP4, nvq.MXFP8)
    wr, wc = nvq.grouped_hybrid_quantize(w2, [N] * G, nvq.NVFP4, nvq.MXFP8)
    y2 = nvq.grouped_gemm_rows(xr, wr, sizes, N, b_col_groups=False)
    dr, dc = nvq.grouped_hybrid_quantize(dy, sizes, nvq.MXFP8, nvq.MXFP8)
    dx2 = nvq.grouped_gemm_rows(dr, wc, sizes, N, b_col_groups=True)
    dw2 = nvq.grouped_gemm_wgrad(dc, xc, sizes)
    torch.cuda.synchronize()

    assert y.shape == (T, N) and dx.shape == (T, K) and dw.shape == (G, N, K)
    assert torch.equal(y, y2)
    assert torch.equal(dx, dx2)
    assert torch.equal(dw, dw2)
    assert torch.count_nonzero(dw[1]) == 0
    for name, a, b in (("x_row", fb["x_row"], xr), ("w_row", fb["w_row"], wr), ("x_col", fb["x_col"], xc),
                       ("w_col", fb["w_col"], wc), ("dy_row", bb["dy_row"], dr), ("dy_col", bb["dy_col"], dc)):
        assert torch.equal(a.data, b.data), name
        assert torch.equal(a.scale, b.scale), name
