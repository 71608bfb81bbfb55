"""Helpers for GPU-vs-oracle parity tests (no method arithmetic here)."""
import numpy as np
import torch

import oracle
import mxfp8_block_scaled_bf16_gb300 as nvq


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (CPU numpy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def qt_codes(q: nvq.QTensor) -> np.ndarray:
    """GPU codes as [rows, bytes per row]."""
    per_row = q.cols // 2 if q.fmt in (nvq.NVFP4, nvq.NVFP4_ROWSCALED) else q.cols
    return q.data[: q.rows * per_row].cpu().numpy().reshape(q.rows, per_row)


def qt_scales(q: nvq.QTensor) -> np.ndarray:
    blk = 16 if q.fmt in (nvq.NVFP4, nvq.NVFP4_ROWSCALED) else 32
    n = oracle.swizzled_size(q.rows, q.cols // blk)
    return q.scale[:n].cpu().numpy()


def assert_codes_equal(got: np.ndarray, want: np.ndarray, what: str):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        r, c = bad[0]
        raise AssertionError(f"{what}: {len(bad)} of {want.size} bytes differ; first at {tuple(bad[0])}: "
                             f"got {got[r, c]:#x} want {want[r, c]:#x}")


def assert_scales_equal(q: nvq.QTensor, compact: np.ndarray, what: str):
    want = oracle.scale_swizzle(compact)
    got = qt_scales(q)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{what}: {len(bad)} of {want.size} swizzled scale bytes differ; first at {bad[0]}: "
                             f"got {got[bad[0]]:#x} want {want[bad[0]]:#x}")


def check_nvfp4_row(q, x, A=None, sr=None, what="nvfp4 row"):
    c, s, A = oracle.nvfp4_quantize_rows(bits(x), A=A, sr=sr)
    assert float(q.amax[0].item()) == np.float32(A), f"{what}: amax {q.amax[0].item()} vs {A}"
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s, A


def check_nvfp4_col(q, x, rht=None, sr=None, what="nvfp4 col"):
    c, s, A = oracle.nvfp4_quantize_cols(bits(x), rht_sign=rht, sr=sr)
    assert float(q.amax[0].item()) == np.float32(A), f"{what}: amax {q.amax[0].item()} vs {A}"
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s, A


def check_mxfp8_row(q, x, what="mxfp8 row"):
    c, s = oracle.mxfp8_quantize_rows(bits(x))
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s


def check_mxfp8_col(q, x, what="mxfp8 col"):
    c, s = oracle.mxfp8_quantize_cols(bits(x))
    assert_codes_equal(qt_codes(q), c, what + " codes")
    assert_scales_equal(q, s, what + " scales")
    return c, s


def bf16_from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def assert_gemm_close(got: torch.Tensor, ref64: np.ndarray, what: str, tol: float = 1e-3, ulp_frac: float = 0.999):
    """fp32 output: relative Frobenius error <= tol against the fp64 oracle.
    bf16 output: relative Frobenius error <= tol against the oracle rounded
    once to bf16, and >= ulp_frac of elements within one bf16 ulp of it."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    if got.dtype == torch.float32:
        ref = ref64
    else:
        ref = bf16_from_bits(oracle.to_bf16_rne(ref64)).float().numpy().astype(np.float64)
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(g - ref) / (nrm if nrm > 0 else 1.0)
    assert rel <= tol, f"{what}: relative Frobenius error {rel:.3e} > {tol}"
    if got.dtype == torch.bfloat16:
        gb = bits(got.reshape(ref.shape)).astype(np.int32)
        rb = oracle.to_bf16_rne(ref64).astype(np.int32)
        # ulp distance on the sign-magnitude bf16 encoding
        def ordered(v):
            return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)
        ulps = np.abs(ordered(gb) - ordered(rb))
        frac = np.mean(ulps <= 1)
        assert frac >= ulp_frac, f"{what}: only {frac:.5f} of elements within 1 bf16 ulp"
    return rel


def sample_positions(R, C, n, seed, line=None):
    """n random (row, col) positions of an R x C output plus one row and one
    column (the first `line` entries of each, all of them when line is None)."""
    rng = np.random.default_rng(seed)
    r = rng.integers(0, R, n)
    c = rng.integers(0, C, n)
    row = int(rng.integers(0, R))
    col = int(rng.integers(0, C))
    lc = C if line is None else min(C, line)
    lr = R if line is None else min(R, line)
    rows = np.concatenate([r, np.full(lc, row), np.arange(lr)])
    cols = np.concatenate([c, np.arange(lc), np.full(lr, col)])
    return rows, cols


def check_sampled_gemm(got: torch.Tensor, fmt, a, b, K, rows, cols, what, tol=1e-3):
    """got: bf16 GPU output (any device); a, b: oracle operands (codes, compact
    scales, amax) of A [R][K] and B [C][K] in format fmt (1 NVFP4, 2 MXFP8).
    The oracle computes each sampled output from its own operands in fp64; the
    GPU values must be within relative Frobenius error tol of it rounded once to
    bf16, and >= 99.9% of them within one bf16 ulp."""
    ga = oracle.nvfp4_g(a[2]) if fmt == 1 else 1.0
    gb = oracle.nvfp4_g(b[2]) if fmt == 1 else 1.0
    ref = oracle.gemm_tn_sampled(fmt, a[0], a[1], ga, b[0], b[1], gb, K, rows, cols)
    sel = got[torch.from_numpy(rows).to(got.device), torch.from_numpy(cols).to(got.device)].cpu()
    g = sel.float().numpy().astype(np.float64)
    refb = bf16_from_bits(oracle.to_bf16_rne(ref)).float().numpy().astype(np.float64)
    nrm = np.linalg.norm(refb)
    rel = np.linalg.norm(g - refb) / (nrm if nrm > 0 else 1.0)
    assert rel <= tol, f"{what}: sampled relative Frobenius error {rel:.3e}"
    gb_ = bits(sel).astype(np.int32)
    rb = oracle.to_bf16_rne(ref).astype(np.int32)

    def ordered(v):
        return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)

    frac = np.mean(np.abs(ordered(gb_) - ordered(rb)) <= 1)
    assert frac >= 0.999, f"{what}: {frac:.5f} of sampled outputs within 1 bf16 ulp"
    return rel
