"""Pins of the oracle's Philox4x32-10 generator and its stochastic rounding.

"Add an NVFP4 quantization converter", section "What changed": stochastic
rounding is keyed by a per-rank Philox seed and is unbiased.  The generator is
pinned against an independent implementation (Triton's Philox, run by its
CPU interpreter); unbiasedness is checked exactly by enumerating every 16-bit
random draw, and statistically over the counter stream.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle

_TRITON_SCRIPT = textwrap.dedent("""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import torch, triton, triton.language as tl

    @triton.jit
    def k(c_ptr, key_ptr, out_ptr, n: tl.constexpr):
        i = tl.arange(0, n)
        c0 = tl.load(c_ptr + 4 * i + 0).to(tl.uint32, bitcast=True)
        c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32, bitcast=True)
        c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32, bitcast=True)
        c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32, bitcast=True)
        k0 = tl.load(key_ptr + 2 * i + 0).to(tl.uint32, bitcast=True)
        k1 = tl.load(key_ptr + 2 * i + 1).to(tl.uint32, bitcast=True)
        a, b, c, d = tl.philox_impl(c0, c1, c2, c3, k0, k1, 10)
        tl.store(out_ptr + 4 * i + 0, a.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 1, b.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 2, c.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 3, d.to(tl.int32, bitcast=True))

    data = json.load(sys.stdin)
    c = torch.tensor(data["ctr"], dtype=torch.int64).to(torch.int32)
    kk = torch.tensor(data["key"], dtype=torch.int64).to(torch.int32)
    n = c.numel() // 4
    out = torch.zeros(4 * n, dtype=torch.int32)
    k[(1,)](c, kk, out, n)
    print(json.dumps([int(v) & 0xFFFFFFFF for v in out.tolist()]))
""")


def _triton_philox(ctrs, keys):
    pytest.importorskip("triton")
    import json
    n = len(ctrs)
    n2 = 1 << max(0, (n - 1).bit_length())  # the interpreter wants a power-of-two block
    ctrs = np.concatenate([ctrs, np.zeros((n2 - n, 4), np.uint32)])
    keys = np.concatenate([keys, np.zeros((n2 - n, 2), np.uint32)])
    inp = json.dumps({"ctr": [int(v) - (1 << 32) if v >= (1 << 31) else int(v) for v in ctrs.reshape(-1)],
                      "key": [int(v) - (1 << 32) if v >= (1 << 31) else int(v) for v in keys.reshape(-1)]})
    env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=inp, capture_output=True,
                       text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1])
    return np.array(json.loads(r.stdout.strip().splitlines()[-1]), dtype=np.uint32).reshape(-1, 4)[:n]


def test_philox_matches_independent_implementation():
    rng = np.random.default_rng(2024)
    n = 256
    ctrs = rng.integers(0, 1 << 32, (n, 4), dtype=np.uint64).astype(np.uint32)
    keys = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    ctrs[0] = 0
    keys[0] = 0
    ctrs[1] = 0xFFFFFFFF
    keys[1] = 0xFFFFFFFF
    want = _triton_philox(ctrs, keys)
    got = np.stack([oracle.philox4x32_10(ctrs[i], keys[i]) for i in range(n)])
    assert np.array_equal(got, want)


def test_sr_bits_stream_layout():
    """16-bit field of element L = word (L&7)>>1, half L&1 of the Philox block
    at counter (lo32(L>>3), hi32(L>>3), direction, offset), key = seed words."""
    seed = -(2 ** 63) + 987654321123  # any int64 (drawn over the full range on the page)
    useed = seed & ((1 << 64) - 1)
    key = np.array([useed & 0xFFFFFFFF, useed >> 32], dtype=np.uint32)
    Ls = [0, 1, 2, 3, 7, 8, 15, 16, (1 << 35) + 5, (1 << 40) + 3]
    ctrs = np.array([[(L >> 3) & 0xFFFFFFFF, (L >> 3) >> 32, d, off]
                     for L in Ls for d in (0, 1) for off in (0, 3)], dtype=np.uint32)
    keys = np.tile(key, (len(ctrs), 1))
    blocks = _triton_philox(ctrs, keys)
    i = 0
    for L in Ls:
        for d in (0, 1):
            for off in (0, 3):
                w = blocks[i]
                want = (int(w[(L & 7) >> 1]) >> (16 * (L & 1))) & 0xFFFF
                assert oracle.sr_bits(seed, off, d, L) == want
                i += 1


@pytest.mark.parametrize("v", [0.1, 0.3, 0.5, 0.75, 1.2, 1.9, 2.25, 2.7, 3.3, 4.5, 5.99, -0.37, -3.1])
def test_sr_exactly_unbiased_over_all_draws(v):
    v = float(np.float32(v))
    vals = np.array([oracle.e2m1_decode(oracle.e2m1_encode_sr(v, r)) for r in range(65536)])
    mean = vals.mean()
    a = abs(v)
    q = 0.5 if a < 2 else (1.0 if a < 4 else 2.0)
    lo = np.floor(a / q) * q
    # each draw gives one of the two neighbours
    assert set(np.abs(vals)) <= {lo, lo + q}
    # P(up) = ceil(frac * 2^16) / 2^16, so the bias is below 2^-16 of a spacing
    assert abs(mean - v) <= q * 2.0 ** -16 + 1e-12
    frac16 = (a - lo) / q * 65536
    if frac16 == int(frac16):
        assert mean == v


def test_sr_exact_grid_values_never_move():
    for c in range(8):
        m = oracle.e2m1_decode(c)
        for r in (0, 1, 32767, 65535):
            assert oracle.e2m1_decode(oracle.e2m1_encode_sr(m, r)) == m


def test_sr_saturates():
    assert oracle.e2m1_encode_sr(6.5, 0) == 7
    assert oracle.e2m1_encode_sr(-100.0, 65535) == 15


def test_sr_statistical_unbiasedness_over_counter_stream():
    """The whole rowwise SR quantizer is unbiased: the mean of the dequantized
    values over many seeds converges to the input within 4 sigma."""
    x = np.array([[0.3, -1.1, 2.6, 4.9, 0.05, -5.5, 1.7, 3.2] * 2], dtype=np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 bit patterns
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    n = 600
    acc = np.zeros(16)
    acc2 = np.zeros(16)
    A = float(np.abs(xf).max())
    for s in range(n):
        c, sc, _ = oracle.nvfp4_quantize_rows(xb, A=A, sr=(s * 7919 + 1, 0))
        d = oracle.nvfp4_dequant(c, sc, oracle.nvfp4_g(A))[0]
        acc += d
        acc2 += d * d
    mean = acc / n
    var = np.maximum(acc2 / n - mean ** 2, 1e-30)
    assert np.all(np.abs(mean - xf[0]) <= 4 * np.sqrt(var / n) + 1e-6)
