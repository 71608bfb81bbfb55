"""Pins of the oracle's element/scale formats against brute force and fixtures.

The format definitions follow the OCP MX v1.0 (E2M1, E8M0) and OFP8 (E4M3)
specifications; the pages only name the formats ("Add an NVFP4 quantization
converter", review thread on "rowwise"; "Hybrid quantization", mxfp8 storage
review).  Each check below uses a method independent of the oracle's code:
enumeration of the decoded code tables with an explicit nearest/tie rule.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        v, c = line.split()
        rows.append((float(v), int(c)))
    return rows


def _all_bf16_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    return f[np.isfinite(f)]


def _brute_nearest(values, codes, decoded):
    """Nearest code by exhaustive search; ties -> the code whose mantissa LSB
    is 0; the sign of the input is kept (a negative value rounding to zero
    gets the negative-zero code).  ``codes`` are non-negative magnitudes."""
    mags = np.array(decoded, dtype=np.float64)
    out = []
    for v in values:
        a = abs(float(v))
        if a >= mags.max():  # satfinite: at or beyond the largest magnitude
            out.append(codes[int(np.argmax(mags))])
            continue
        d = np.abs(mags - a)
        best = d.min()
        cand = [codes[i] for i in np.nonzero(d == best)[0]]
        if len(cand) > 1:
            cand = [c for c in cand if c & 1 == 0]
        assert len(cand) == 1
        out.append(cand[0])
    return np.array(out)


def test_e2m1_decode_table():
    expect = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert oracle.e2m1_decode(c) == expect[c]
        assert oracle.e2m1_decode(c | 8) == -expect[c]


def test_e4m3_decode_table():
    # OFP8 E4M3: bias 7, subnormal m/8 * 2^-6, NaN only at S.1111.111
    vals = [oracle.e4m3_decode(c) for c in range(256)]
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    finite = [v for i, v in enumerate(vals) if i not in (0x7F, 0xFF)]
    assert max(finite) == 448.0 and min(finite) == -448.0
    assert vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6
    pos = sorted(set(v for v in finite if v >= 0))
    assert len(pos) == 127  # 0 plus 126 positive finite values


def test_e8m0_decode():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(oracle.e8m0_decode(255))


@pytest.mark.parametrize("v,code", _fixture("e2m1_ties.txt"))
def test_e2m1_golden(v, code):
    assert oracle.e2m1_encode_rn(v) == code


@pytest.mark.parametrize("v,code", _fixture("e4m3_points.txt"))
def test_e4m3_golden(v, code):
    assert oracle.e4m3_encode_rn(v) == code


def test_e2m1_encode_exhaustive_bf16():
    vals = _all_bf16_finite()
    decoded = [oracle.e2m1_decode(c) for c in range(8)]
    want = _brute_nearest(vals, list(range(8)), decoded)
    want = want | np.where(np.signbit(vals), 8, 0)
    got = np.array([oracle.e2m1_encode_rn(float(v)) for v in vals])
    assert np.array_equal(got, want)


def test_e4m3_encode_exhaustive_bf16_and_random_fp32():
    rng = np.random.default_rng(11)
    rnd = (rng.standard_normal(100_000) * np.exp2(rng.integers(-14, 10, 100_000))).astype(np.float32)
    vals = np.concatenate([_all_bf16_finite(), rnd])
    codes = [c for c in range(127)]  # non-negative finite codes 0..0x7E
    decoded = [oracle.e4m3_decode(c) for c in codes]
    want = _brute_nearest(vals, codes, decoded) | np.where(np.signbit(vals), 0x80, 0)
    got = np.array([oracle.e4m3_encode_rn(float(v)) for v in vals])
    assert np.array_equal(got, want)


def test_e4m3_matches_torch_cast_on_representable_range():
    # torch.float8_e4m3fn casts with round-to-nearest-even; saturation differs
    # (torch gives NaN above 464), so compare inside the finite range only.
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(50_000) * np.exp2(rng.integers(-12, 8, 50_000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode_rn(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, t)


def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(9)
    v = (rng.standard_normal(20_000) * np.exp2(rng.integers(-30, 30, 20_000))).astype(np.float32)
    # add exact ties (fp32 values halfway between bf16 neighbours)
    ties = ((rng.integers(0, 1 << 15, 2000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    v = np.concatenate([v, ties[np.isfinite(ties)]])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.to_bf16_rne(v.astype(np.float64))
    assert np.array_equal(got, want)
