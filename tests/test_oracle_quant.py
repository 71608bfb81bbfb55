"""Pins of the oracle's NVFP4 / MXFP8 block quantizers and the scale layout.

Pages: "Add an NVFP4 quantization converter" (NVFP4 = FP32 tensor scale plus
an E4M3 scale per 1x16 block; RHT and SR on the wgrad operands) and "Hybrid
quantization" (MXFP8 in 32-element blocks with E8M0 scales; ceil(M/32)
columnwise scale rows).  The checks use exact round trips of representable
values, nearest-point searches over each block's grid, transposition and
Hadamard identities computed with scipy, and the ceil-vs-floor scale count.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from mxfp8_block_scaled_bf16_gb300.inputs import rht_sign_vector, student_t3_outliers

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _bits(xf):
    """fp32 values that are exactly bf16 -> bf16 bit patterns."""
    xf = np.ascontiguousarray(xf, dtype=np.float32)
    b = xf.view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def _f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rand_bf16(M, K, seed=0, std=1.0):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(M, K, generator=g) * std).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_exact_round_trip_of_representable_blocks():
    """Blocks of E2M1 grid values scaled by 2^(p-j) with block max 6*2^(p-j):
    the scale is exactly 448*2^-j and every code is the grid value itself, so
    decoding gives x back up to the fp32 rounding of g = A/2688."""
    rng = np.random.default_rng(0)
    M, K, p = 32, 256, 3
    x = np.zeros((M, K), np.float32)
    want_codes = np.zeros((M, K), np.uint8)
    want_scales = np.zeros((M, K // 16), np.uint8)
    for i in range(M):
        for j in range(K // 16):
            jj = (i + j) % 10  # block-scale exponent offset
            c = rng.choice(E2M1, 16) * rng.choice([-1, 1], 16)
            c[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            x[i, 16 * j:16 * j + 16] = c * 2.0 ** (p - jj)
            want_codes[i, 16 * j:16 * j + 16] = [
                (8 if np.signbit(v) else 0) | int(np.nonzero(E2M1 == abs(v))[0][0]) for v in c]
            want_scales[i, j] = oracle.e4m3_encode_rn(448.0 * 2.0 ** -jj)
            assert oracle.e4m3_decode(int(want_scales[i, j])) == 448.0 * 2.0 ** -jj
    xb = _bits(x)
    codes, scales, A = oracle.nvfp4_quantize_rows(xb)
    assert A == 6.0 * 2 ** p
    assert np.array_equal(scales, want_scales)
    # packing: two codes per byte, low nibble = even element
    assert np.array_equal(codes, want_codes[:, 0::2] | (want_codes[:, 1::2] << 4))
    deq = oracle.nvfp4_dequant(codes, scales, oracle.nvfp4_g(A))
    np.testing.assert_allclose(deq, x.astype(np.float64), rtol=1e-7, atol=0)


def test_nvfp4_rows_are_nearest_on_block_grid():
    """Every decoded element is a nearest point of its block's grid
    {E2M1 values * E4M3(S) * g} (up to fp32 rounding of the encode factor),
    and the stored scale is a nearest E4M3 value to b*448/A."""
    xb = _rand_bf16(64, 512, seed=1)
    xf = _f32(xb).astype(np.float64)
    codes, scales, A = oracle.nvfp4_quantize_rows(xb)
    g = oracle.nvfp4_g(A)
    deq = oracle.nvfp4_dequant(codes, scales, g)
    e4m3 = np.array([oracle.e4m3_decode(c) for c in range(127)])
    for i in range(64):
        for j in range(32):
            blk = xf[i, 16 * j:16 * j + 16]
            b = np.abs(blk).max()
            S = oracle.e4m3_decode(int(scales[i, j]))
            target = b * 448.0 / A
            assert abs(S - target) <= np.abs(e4m3 - target).min() * (1 + 1e-6) + 1e-12
            grid = E2M1 * S * g
            for t in range(16):
                d = np.abs(grid - abs(blk[t])).min()
                assert abs(abs(deq[i, 16 * j + t]) - abs(blk[t])) <= d + 1e-6 * S * g
                assert deq[i, 16 * j + t] == 0 or np.sign(deq[i, 16 * j + t]) == np.sign(blk[t])


def test_nvfp4_cols_equal_rows_of_transpose():
    xb = _rand_bf16(96, 64, seed=2)
    cc, cs, A1 = oracle.nvfp4_quantize_cols(xb)
    rc, rs, A2 = oracle.nvfp4_quantize_rows(np.ascontiguousarray(xb.T))
    assert A1 == A2
    assert np.array_equal(cc, rc) and np.array_equal(cs, rs)


def test_nvfp4_cols_ragged_tail_is_zero_padded():
    xb = _rand_bf16(40, 32, seed=3)
    cc, cs, A = oracle.nvfp4_quantize_cols(xb)
    assert cc.shape == (32, 24) and cs.shape == (32, 3)
    pad = np.zeros((48, 32), np.uint16)
    pad[:40] = xb
    pc, ps, A2 = oracle.nvfp4_quantize_cols(pad)
    assert A == A2 and np.array_equal(cc, pc) and np.array_equal(cs, ps)


def _rht_lattice_input(M, K, sign, seed):
    """x whose blocks are s * (sparse small-integer vectors) / 4: both x and
    T(x) are exact in bf16 and the fp32 butterfly is exact."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, K), np.float32)
    for k in range(K):
        for j in range(M // 16):
            y = np.zeros(16)
            idx = rng.choice(16, 3, replace=False)
            y[idx] = rng.integers(-6, 7, 3)
            x[16 * j:16 * j + 16, k] = sign * y / 4.0
    return x


def test_nvfp4_cols_rht_equals_plain_cols_of_transformed_input():
    s = rht_sign_vector(7)
    H = scipy.linalg.hadamard(16).astype(np.float64)
    M, K = 64, 32
    x = _rht_lattice_input(M, K, s, seed=5)
    tx = np.zeros_like(x, dtype=np.float64)
    for j in range(M // 16):
        blk = x[16 * j:16 * j + 16].astype(np.float64)  # [16, K]
        tx[16 * j:16 * j + 16] = 0.25 * H @ (s[:, None] * blk)
    xb, txb = _bits(x), _bits(tx.astype(np.float32))
    A_rht = oracle.amax_rht_col(xb, s)
    assert A_rht == np.abs(tx).max()
    c1, s1, _ = oracle.nvfp4_quantize_cols(xb, rht_sign=s)
    c2, s2, _ = oracle.nvfp4_quantize_cols(txb)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_nvfp4_sr_picks_grid_neighbours():
    xb = _rand_bf16(32, 64, seed=6)
    xf = _f32(xb).astype(np.float64)
    codes, scales, A = oracle.nvfp4_quantize_rows(xb, sr=(1234, 0))
    rc, rs, _ = oracle.nvfp4_quantize_rows(xb)
    assert np.array_equal(scales, rs)  # scales are always round-to-nearest
    g = oracle.nvfp4_g(A)
    deq = oracle.nvfp4_dequant(codes, scales, g)
    for i in range(32):
        for j in range(4):
            S = oracle.e4m3_decode(int(scales[i, j]))
            grid = E2M1 * S * g
            for t in range(16):
                a = abs(xf[i, 16 * j + t])
                below = grid[grid <= a * (1 + 1e-6)].max()
                above = grid[grid >= a * (1 - 1e-6)].min() if a <= grid[-1] else grid[-1]
                assert abs(deq[i, 16 * j + t]) in (below, above)
    assert not np.array_equal(codes, rc)  # SR changes some codes
    c2, _, _ = oracle.nvfp4_quantize_rows(xb, sr=(1234, 0))
    assert np.array_equal(codes, c2)  # deterministic under the same key
    c3, _, _ = oracle.nvfp4_quantize_rows(xb, sr=(1235, 0))
    assert not np.array_equal(codes, c3)


def test_nvfp4_zero_tensor_and_zero_blocks():
    xb = np.zeros((16, 32), np.uint16)
    c, s, A = oracle.nvfp4_quantize_rows(xb)
    assert A == 0.0 and not c.any() and not s.any()
    assert oracle.nvfp4_s_enc(0.0) == 1.0
    x = np.zeros((16, 32), np.float32)
    x[0, 0] = 3.0
    c, s, A = oracle.nvfp4_quantize_rows(_bits(x))
    assert s[0, 0] == 0x7E and not s[1:].any() and not s[0, 1:].any()


def test_amax_matches_numpy():
    xb = _bits(_f32(student_t3_outliers(64, 256).view(torch.int16).numpy().view(np.uint16)))
    assert oracle.amax(xb) == np.abs(_f32(xb)).max()


# ------------------------------------------------------------------ MXFP8
def test_mxfp8_exact_round_trip_of_representable_blocks():
    rng = np.random.default_rng(7)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(127)])
    M, K = 16, 128
    x = np.zeros((M, K), np.float32)
    for i in range(M):
        for j in range(K // 32):
            p = int(rng.integers(-20, 20))
            c = rng.choice(e4[e4 <= 448], 32) * rng.choice([-1, 1], 32)
            c[rng.integers(32)] = rng.choice([256.0, 288.0, 448.0])  # block max in [256, 448]
            x[i, 32 * j:32 * j + 32] = c * 2.0 ** p
    xb = _bits(x)
    codes, scales = oracle.mxfp8_quantize_rows(xb)
    assert np.array_equal(oracle.mxfp8_dequant(codes, scales), x.astype(np.float64))


def test_mxfp8_scale_is_power_of_two_floor():
    """E8M0 scale 2^e with 256 <= b / 2^e < 512 (largest power of two not
    above b, divided by 2^8 = the largest power of two of E4M3)."""
    xb = _rand_bf16(32, 256, seed=8)
    xf = _f32(xb).astype(np.float64)
    _, scales = oracle.mxfp8_quantize_rows(xb)
    for i in range(32):
        for j in range(8):
            b = np.abs(xf[i, 32 * j:32 * j + 32]).max()
            r = b / oracle.e8m0_decode(int(scales[i, j]))
            assert 256 <= r < 512


def test_mxfp8_elements_nearest_or_saturated():
    xb = _rand_bf16(16, 128, seed=9)
    xf = _f32(xb).astype(np.float64)
    codes, scales = oracle.mxfp8_quantize_rows(xb)
    deq = oracle.mxfp8_dequant(codes, scales)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(127)])
    for i in range(16):
        for j in range(4):
            sc = oracle.e8m0_decode(int(scales[i, j]))
            grid = e4 * sc
            for t in range(32):
                a = abs(xf[i, 32 * j + t])
                if a >= 448 * sc:
                    assert abs(deq[i, 32 * j + t]) == 448 * sc
                else:
                    assert abs(abs(deq[i, 32 * j + t]) - a) == np.abs(grid - a).min()


@pytest.mark.parametrize("M", [48, 33, 64, 1])
def test_mxfp8_colwise_scale_count_is_ceil(M):
    xb = _rand_bf16(M, 32, seed=10)
    codes, scales = oracle.mxfp8_quantize_cols(xb)
    assert scales.shape == (32, -(-M // 32))
    if M % 32:
        assert scales.shape[1] != M // 32  # floor would drop the tail block
        # the tail block's scale is a real scale of the tail rows, not padding
        tail = _f32(xb[(M // 32) * 32:]).astype(np.float64)
        b = np.abs(tail).max(axis=0)
        for k in range(32):
            if b[k] > 0:
                r = b[k] / oracle.e8m0_decode(int(scales[k, -1]))
                assert 256 <= r < 512


def test_mxfp8_cols_equal_rows_of_transpose():
    xb = _rand_bf16(64, 96, seed=11)
    cc, cs = oracle.mxfp8_quantize_cols(xb)
    rc, rs = oracle.mxfp8_quantize_rows(np.ascontiguousarray(xb.T))
    assert np.array_equal(cc, rc) and np.array_equal(cs, rs)


# ------------------------------------------------------------------ scale layout
def test_scale_swizzle_is_padded_bijection():
    R, C = 200, 9
    rng = np.random.default_rng(12)
    compact = rng.integers(1, 255, (R, C)).astype(np.uint8)
    swz = oracle.scale_swizzle(compact)
    assert swz.size == 256 * 12
    assert np.count_nonzero(swz) == R * C  # pads are zero, nothing overwritten
    assert np.array_equal(oracle.scale_unswizzle(swz, R, C), compact)


def test_scale_swizzle_known_positions():
    """128x4 tiles of 512 B; inside a tile row r sits at (r%32)*16 + (r/32)*4."""
    R, C = 256, 8
    pos = {}
    for r, c in [(0, 0), (0, 1), (1, 0), (32, 0), (96, 3), (127, 3), (0, 4), (128, 0)]:
        compact = np.zeros((R, C), np.uint8)
        compact[r, c] = 1
        pos[(r, c)] = int(np.nonzero(oracle.scale_swizzle(compact))[0][0])
    assert pos == {(0, 0): 0, (0, 1): 1, (1, 0): 16, (32, 0): 4, (96, 3): 15, (127, 3): 511,
                   (0, 4): 512, (128, 0): 1024}


def test_offset_variants_are_slices_of_the_whole_tensor():
    """Quantizing rows r0.. of a tensor with its amax and index offset gives
    exactly the rows (or, columnwise, the contraction columns) of the
    whole-tensor quantization, stochastic-rounding draws included."""
    import torch
    from mxfp8_block_scaled_bf16_gb300 import inputs
    x = inputs.normal_bf16((112, 48), 1.0, torch.Generator().manual_seed(8))
    sign = inputs.rht_sign_vector()
    for sr in (None, (99, 3)):
        c, s, A = oracle.nvfp4_quantize_rows(x, sr=sr)
        for r0, n in ((0, 16), (32, 48), (96, 16), (40, 7)):
            c2, s2 = oracle.nvfp4_quantize_rows_at(x[r0:r0 + n], A, r0, sr=sr)
            assert np.array_equal(c[r0:r0 + n], c2) and np.array_equal(s[r0:r0 + n], s2)
        for rht in (None, sign):
            c, s, A = oracle.nvfp4_quantize_cols(x, rht_sign=rht, sr=sr)
            for r0, n in ((0, 16), (32, 48), (96, 16)):
                c2, s2 = oracle.nvfp4_quantize_cols_at(x[r0:r0 + n], A, r0, 112, rht_sign=rht, sr=sr)
                assert np.array_equal(c[:, r0 // 2:(r0 + n) // 2], c2)
                assert np.array_equal(s[:, r0 // 16:(r0 + n) // 16], s2)
