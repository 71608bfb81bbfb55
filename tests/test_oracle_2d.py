"""Pins of the oracle's NVFP4 2D (16 x 16) columnwise block scaling ("Hybrid
quantization", timeline: "[Common] Enable NVFP4 2D block scaling in columnwise
only"), read as one E4M3 scale per 16 x 16 tile shared by the tile's sixteen
columnwise 1 x 16 blocks."""
import numpy as np
import torch

import oracle
from mxfp8_block_scaled_bf16_gb300 import inputs


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _deq_cols(c, s, A):
    return oracle.nvfp4_dequant(c, s, oracle.nvfp4_g(A))


def test_scale_is_shared_by_each_tile():
    x = inputs.student_t3_outliers(64, 96)
    c, s, A = oracle.nvfp4_quantize_cols_2d(x)
    for k0 in range(0, 96, 16):
        assert np.all(s[k0:k0 + 16] == s[k0])  # the 16 columns of a tile share the scale of each row block


def test_tile_scaling_is_the_same_for_x_and_its_transpose():
    """A 16 x 16 tile is scaled as one unit, so quantizing x's columns and
    x^T's columns dequantize to the same values (transposed) -- the property
    that makes a weight's forward and backward copies agree."""
    x = inputs.normal_bf16((64, 48), 1.0, torch.Generator().manual_seed(3))
    c1, s1, A1 = oracle.nvfp4_quantize_cols_2d(x)
    c2, s2, A2 = oracle.nvfp4_quantize_cols_2d(x.t().contiguous())
    assert A1 == A2
    d1 = _deq_cols(c1, s1, A1)  # [K][M] = quantized x^T
    d2 = _deq_cols(c2, s2, A2)  # [M][K] = quantized x
    assert np.array_equal(d1, d2.T)


def test_reduces_to_the_1d_blocks_when_a_tile_has_one_nonzero_column():
    x = torch.zeros(48, 64, dtype=torch.float32)
    g = torch.Generator().manual_seed(4)
    for c0 in range(0, 64, 16):
        x[:, c0 + int(torch.randint(0, 16, (1,), generator=g))] = torch.randn(48, generator=g)
    x = x.to(torch.bfloat16)
    c2, s2, A2 = oracle.nvfp4_quantize_cols_2d(x)
    c1, s1, A1 = oracle.nvfp4_quantize_cols(x)
    assert A1 == A2
    nz = np.abs(_bits(x).astype(np.int32) & 0x7FFF).reshape(3, 16, 64).max(axis=1).T > 0  # [K][row blocks]
    assert np.array_equal(c2, c1)  # zero columns encode to zero either way
    assert np.array_equal(s2[nz], s1[nz])


def test_representable_tiles_round_trip():
    """Tiles of E2M1 grid values times a power of two with a 6 in every tile
    (tensor amax 2688) dequantize back exactly."""
    rng = np.random.default_rng(5)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    x = np.zeros((32, 32))
    for i in range(0, 32, 16):
        for j in range(0, 32, 16):
            t = rng.choice(grid, (16, 16)) * rng.choice([-1, 1], (16, 16))
            t[rng.integers(16), rng.integers(16)] = 6.0
            # tile (0, 0) at scale 448 holds the tensor amax 6 * 448 = 2688
            x[i:i + 16, j:j + 16] = t * (448.0 if i == j == 0 else 2.0 ** int(rng.integers(-2, 2)))
    xt = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    c, s, A = oracle.nvfp4_quantize_cols_2d(xt)
    assert A == 2688.0
    assert np.array_equal(_deq_cols(c, s, A), x.T)
