"""CPU oracle for the block-scaled quantize + GEMM path (TEST INFRASTRUCTURE).

Only the tests, the smoke check and the benchmark's CPU-baseline / reference
leg use this package.  The library never imports it, and it imports nothing
from the library.  The arithmetic lives in ``oracle.c`` (plain C, fp32 with
round-to-nearest-even and no contraction, fp64 GEMM accumulation); this file
only compiles it and marshals numpy arrays.

Every function cites the page it follows in ``oracle.c``.  Readings of steps
the pages leave open are marked READING there.  Parity pins live in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (portable C99, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=gnu99", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, u32, f32, f64, i32 = (ctypes.c_int64, ctypes.c_uint32, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_int)
            sig = {
                "orc_bf16_to_f32": (f32, [ctypes.c_uint16]),
                "orc_e2m1_decode": (f64, [ctypes.c_uint8]),
                "orc_e4m3_decode": (f64, [ctypes.c_uint8]),
                "orc_e8m0_decode": (f64, [ctypes.c_uint8]),
                "orc_e2m1_encode_rn": (ctypes.c_uint8, [f32]),
                "orc_e4m3_encode_rn": (ctypes.c_uint8, [f32]),
                "orc_e2m1_encode_sr": (ctypes.c_uint8, [f32, u32]),
                "orc_philox4x32_10": (None, [P, P, P]),
                "orc_sr_bits": (u32, [i64, u32, i32, ctypes.c_uint64]),
                "orc_rht16": (None, [P, P]),
                "orc_amax": (f32, [P, i64, i64, i64]),
                "orc_amax_rht_col": (f32, [P, i64, i64, i64, P]),
                "orc_nvfp4_s_enc": (f32, [f32]),
                "orc_nvfp4_g": (f32, [f32]),
                "orc_nvfp4_quantize_rows": (None, [P, i64, i64, i64, f32, i32, i64, u32, P, P]),
                "orc_nvfp4_quantize_cols": (None, [P, i64, i64, i64, f32, P, i32, i64, u32, P, P]),
                "orc_nvfp4_quantize_rows_at": (None, [P, i64, i64, i64, f32, i32, i64, u32, i64, P, P]),
                "orc_nvfp4_quantize_cols_at": (None, [P, i64, i64, i64, f32, P, i32, i64, u32, i64, i64, P, P]),
                "orc_mxfp8_quantize_rows": (None, [P, i64, i64, i64, P, P]),
                "orc_mxfp8_quantize_cols": (None, [P, i64, i64, i64, P, P]),
                "orc_swizzled_size": (i64, [i64, i64]),
                "orc_scale_swizzle": (None, [P, i64, i64, P]),
                "orc_scale_unswizzle": (None, [P, i64, i64, P]),
                "orc_nvfp4_dequant": (None, [P, P, i64, i64, f32, P]),
                "orc_mxfp8_dequant": (None, [P, P, i64, i64, P]),
                "orc_gemm_tn_f64": (None, [P, P, i64, i64, i64, f64, P, P]),
                "orc_gemm_tn_sampled": (None, [i32, P, P, f32, P, P, f32, i64, P, i64, P, P, P]),
                "orc_f64_to_bf16_rne": (None, [P, i64, P]),
                "orc_nvfp4_dequant_bf16": (None, [P, P, i64, i64, f32, P]),
                "orc_mxfp8_dequant_bf16": (None, [P, P, i64, i64, P]),
                "orc_identity_rows": (None, [P, i64, i64, i64, P]),
                "orc_identity_cols": (None, [P, i64, i64, i64, P]),
                "orc_nvfp4_quantize_rows_rowscaled": (None, [P, i64, i64, i64, P, P, P]),
                "orc_nvfp4_quantize_cols_2d": (None, [P, i64, i64, i64, f32, P, P]),
                "orc_nvfp4_dequant_rowscaled": (None, [P, P, i64, i64, P, P]),
                "orc_gemm_tn_sampled_rowscaled": (None, [P, P, P, P, P, f32, i64, i64, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bit patterns."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return x


def _sign(sign) -> np.ndarray:
    s = np.ascontiguousarray(np.asarray(sign, dtype=np.int8).reshape(16))
    if not np.all(np.abs(s) == 1):
        raise ValueError("RHT sign vector must hold 16 values of +-1")
    return s


# ---------------------------------------------------------------- formats
def e2m1_decode(code: int) -> float:
    return _load().orc_e2m1_decode(code)


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(code)


def e8m0_decode(code: int) -> float:
    return _load().orc_e8m0_decode(code)


def e2m1_encode_rn(v: float) -> int:
    return _load().orc_e2m1_encode_rn(v)


def e4m3_encode_rn(v: float) -> int:
    return _load().orc_e4m3_encode_rn(v)


def e2m1_encode_sr(v: float, r16: int) -> int:
    return _load().orc_e2m1_encode_sr(v, r16)


def bf16_to_f32(bits: int) -> float:
    return _load().orc_bf16_to_f32(bits)


# ---------------------------------------------------------------- philox / SR
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bits(seed: int, offset: int, direction: int, L: int) -> int:
    return _load().orc_sr_bits(seed, offset, direction, L)


# ---------------------------------------------------------------- RHT
def rht16(u, sign) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(u, dtype=np.float32).reshape(16)).copy()
    _load().orc_rht16(_p(v), _p(_sign(sign)))
    return v


# ---------------------------------------------------------------- amax
def amax(x) -> float:
    xb = _bf16_bits(x)
    M, K = xb.shape
    return _load().orc_amax(_p(xb), M, K, K)


def amax_rht_col(x, sign) -> float:
    xb = _bf16_bits(x)
    M, K = xb.shape
    return _load().orc_amax_rht_col(_p(xb), M, K, K, _p(_sign(sign)))


def nvfp4_s_enc(A: float) -> float:
    return _load().orc_nvfp4_s_enc(A)


def nvfp4_g(A: float) -> float:
    return _load().orc_nvfp4_g(A)


# ---------------------------------------------------------------- quantize
def nvfp4_quantize_rows(x, A: float | None = None, sr=None):
    """Rowwise NVFP4 of bf16 x[M,K] -> (codes u8[M,K/2], scales u8[M,K/16], A).

    ``sr`` is None (round to nearest) or ``(seed, offset)``."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if A is None:
        A = amax(xb)
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    seed, off = (sr if sr is not None else (0, 0))
    _load().orc_nvfp4_quantize_rows(_p(xb), M, K, K, A, int(sr is not None), seed, off,
                                    _p(codes), _p(scales))
    return codes, scales, A


def nvfp4_quantize_cols(x, A: float | None = None, rht_sign=None, sr=None):
    """Columnwise NVFP4 of bf16 x[M,K] -> (codes u8[K,Mp/2], scales u8[K,Mp/16], A),
    Mp = M rounded up to 16; optional RHT along M and SR."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    s = _sign(rht_sign) if rht_sign is not None else None
    if A is None:
        A = amax_rht_col(xb, s) if s is not None else amax(xb)
    nb = (M + 15) // 16
    codes = np.zeros((K, nb * 8), np.uint8)
    scales = np.zeros((K, nb), np.uint8)
    seed, off = (sr if sr is not None else (0, 0))
    _load().orc_nvfp4_quantize_cols(_p(xb), M, K, K, A, _p(s) if s is not None else None,
                                    int(sr is not None), seed, off, _p(codes), _p(scales))
    return codes, scales, A


def nvfp4_quantize_rows_at(x_rows, A: float, row0: int, sr=None):
    """Rowwise NVFP4 of rows row0.. of a larger tensor whose amax is A (the
    stochastic-rounding bits are those of the rows' positions in that tensor)."""
    xb = _bf16_bits(x_rows)
    M, K = xb.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    seed, off = (sr if sr is not None else (0, 0))
    _load().orc_nvfp4_quantize_rows_at(_p(xb), M, K, K, A, int(sr is not None), seed, off, row0,
                                       _p(codes), _p(scales))
    return codes, scales


def nvfp4_quantize_cols_at(x_rows, A: float, row0: int, Mp_total: int, rht_sign=None, sr=None):
    """Columnwise NVFP4 of rows row0.. (row0 % 16 == 0) of a larger tensor whose
    columnwise storage has Mp_total columns and whose (transformed) amax is A:
    returns (codes u8[K, Mp/2], compact scales u8[K, Mp/16]) for those rows."""
    xb = _bf16_bits(x_rows)
    M, K = xb.shape
    if row0 % 16:
        raise ValueError("row0 must be a multiple of 16")
    s = _sign(rht_sign) if rht_sign is not None else None
    nb = (M + 15) // 16
    codes = np.zeros((K, nb * 8), np.uint8)
    scales = np.zeros((K, nb), np.uint8)
    seed, off = (sr if sr is not None else (0, 0))
    _load().orc_nvfp4_quantize_cols_at(_p(xb), M, K, K, A, _p(s) if s is not None else None,
                                       int(sr is not None), seed, off, row0, Mp_total, _p(codes), _p(scales))
    return codes, scales


def mxfp8_quantize_rows(x):
    xb = _bf16_bits(x)
    M, K = xb.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = np.zeros((M, K), np.uint8)
    scales = np.zeros((M, K // 32), np.uint8)
    _load().orc_mxfp8_quantize_rows(_p(xb), M, K, K, _p(codes), _p(scales))
    return codes, scales


def mxfp8_quantize_cols(x):
    xb = _bf16_bits(x)
    M, K = xb.shape
    nb = (M + 31) // 32
    codes = np.zeros((K, nb * 32), np.uint8)
    scales = np.zeros((K, nb), np.uint8)
    _load().orc_mxfp8_quantize_cols(_p(xb), M, K, K, _p(codes), _p(scales))
    return codes, scales


# ---------------------------------------------------------------- scale layout
def scale_swizzle(compact: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(compact, dtype=np.uint8)
    R, C = c.shape
    out = np.zeros(_load().orc_swizzled_size(R, C), np.uint8)
    _load().orc_scale_swizzle(_p(c), R, C, _p(out))
    return out


def scale_unswizzle(swz: np.ndarray, R: int, C: int) -> np.ndarray:
    s = np.ascontiguousarray(np.asarray(swz, dtype=np.uint8).reshape(-1))
    if s.size < _load().orc_swizzled_size(R, C):
        raise ValueError("swizzled buffer too small")
    out = np.zeros((R, C), np.uint8)
    _load().orc_scale_unswizzle(_p(s), R, C, _p(out))
    return out


def swizzled_size(R: int, C: int) -> int:
    return _load().orc_swizzled_size(R, C)


# ---------------------------------------------------------------- dequant / GEMM
def nvfp4_dequant(codes, scales, g: float) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape[0], c.shape[1] * 2
    out = np.zeros((R, C), np.float64)
    _load().orc_nvfp4_dequant(_p(c), _p(s), R, C, g, _p(out))
    return out


def mxfp8_dequant(codes, scales) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape
    out = np.zeros((R, C), np.float64)
    _load().orc_mxfp8_dequant(_p(c), _p(s), R, C, _p(out))
    return out


def gemm_tn_f64(A: np.ndarray, B: np.ndarray, alpha: float = 1.0, bias=None) -> np.ndarray:
    a = np.ascontiguousarray(A, dtype=np.float64)
    b = np.ascontiguousarray(B, dtype=np.float64)
    R, K = a.shape
    Cn, K2 = b.shape
    if K != K2:
        raise ValueError("contraction lengths differ")
    bb = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64).reshape(Cn)
    out = np.zeros((R, Cn), np.float64)
    _load().orc_gemm_tn_f64(_p(a), _p(b), R, Cn, K, alpha, _p(bb) if bb is not None else None,
                            _p(out))
    return out


def gemm_tn_f64_blas(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """out[r, c] = sum_k A[r, k] B[c, k] in fp64 through numpy's matmul (a
    library routine used as the dot-product step, for outputs too large for
    the naive loop of gemm_tn_f64; same definition, different summation order,
    both fp64)."""
    a = np.ascontiguousarray(A, dtype=np.float64)
    b = np.ascontiguousarray(B, dtype=np.float64)
    if a.shape[1] != b.shape[1]:
        raise ValueError("contraction lengths differ")
    return a @ b.T


def gemm_tn_sampled(fmt: int, a_codes, a_scales, g_a, b_codes, b_scales, g_b, K, rows, cols,
                    bias=None) -> np.ndarray:
    """fmt 1 = NVFP4, 2 = MXFP8; compact scales; returns fp64 outputs at (rows[s], cols[s])."""
    ac = np.ascontiguousarray(a_codes, dtype=np.uint8)
    asc = np.ascontiguousarray(a_scales, dtype=np.uint8)
    bc = np.ascontiguousarray(b_codes, dtype=np.uint8)
    bsc = np.ascontiguousarray(b_scales, dtype=np.uint8)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    bb = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    out = np.zeros(r.size, np.float64)
    _load().orc_gemm_tn_sampled(fmt, _p(ac), _p(asc), float(g_a), _p(bc), _p(bsc), float(g_b), K,
                                _p(bb) if bb is not None else None, r.size, _p(r), _p(c),
                                _p(out))
    return out


def to_bf16_rne(v) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16) with a single round to nearest even."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros(a.shape, np.uint16)
    _load().orc_f64_to_bf16_rne(_p(a), a.size, _p(out))
    return out


# ---------------------------------------------------------------- rowwise-dequantized source / identity
def nvfp4_dequant_bf16(codes, scales, A: float) -> np.ndarray:
    """bf16 bit patterns of the dequantized NVFP4 operand (fp32 (E2M1*E4M3)*g, one RNE to bf16)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape[0], c.shape[1] * 2
    out = np.zeros((R, C), np.uint16)
    _load().orc_nvfp4_dequant_bf16(_p(c), _p(s), R, C, A, _p(out))
    return out


def mxfp8_dequant_bf16(codes, scales) -> np.ndarray:
    """bf16 bit patterns of the dequantized MXFP8 operand (E4M3*2^e exact, one RNE to bf16)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape
    out = np.zeros((R, C), np.uint16)
    _load().orc_mxfp8_dequant_bf16(_p(c), _p(s), R, C, _p(out))
    return out


def identity_rows(x) -> np.ndarray:
    xb = _bf16_bits(x)
    M, K = xb.shape
    out = np.zeros((M, K), np.uint16)
    _load().orc_identity_rows(_p(xb), M, K, K, _p(out))
    return out


def identity_cols(x) -> np.ndarray:
    """x[M,K] -> out[K, Mp] (Mp = M rounded up to 16, pad columns zero)."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    out = np.zeros((K, (M + 15) // 16 * 16), np.uint16)
    _load().orc_identity_cols(_p(xb), M, K, K, _p(out))
    return out


def rowwise_dequantized(x, row_fmt: int, sr=None):
    """The columnwise source of columnwise_source = "rowwise_dequantized": the
    rowwise quantization of x (NVFP4 = 1 with its tensor amax, MXFP8 = 2)
    dequantized to bf16.  Returns (bf16 bits [M,K], rowwise operand)."""
    if row_fmt == 1:
        c, s, A = nvfp4_quantize_rows(x, sr=sr)
        return nvfp4_dequant_bf16(c, s, A), (c, s, A)
    if row_fmt == 2:
        c, s = mxfp8_quantize_rows(x)
        return mxfp8_dequant_bf16(c, s), (c, s)
    raise ValueError("the rowwise direction must be NVFP4 (1) or MXFP8 (2)")


# ---------------------------------------------------------------- row-scaled NVFP4
def nvfp4_quantize_rows_rowscaled(x):
    """Row-scaled NVFP4 of bf16 x[M,K] (a per-row FP32 outer scale) ->
    (codes u8[M,K/2], compact scales u8[M,K/16], per-row amax f32[M])."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    amax_rows = np.zeros(M, np.float32)
    _load().orc_nvfp4_quantize_rows_rowscaled(_p(xb), M, K, K, _p(codes), _p(scales), _p(amax_rows))
    return codes, scales, amax_rows


def nvfp4_dequant_rowscaled(codes, scales, amax_rows) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    a = np.ascontiguousarray(amax_rows, dtype=np.float32)
    R, C = c.shape[0], c.shape[1] * 2
    out = np.zeros((R, C), np.float64)
    _load().orc_nvfp4_dequant_rowscaled(_p(c), _p(s), R, C, _p(a), _p(out))
    return out


def gemm_tn_sampled_rowscaled(a_codes, a_scales, a_amax_rows, b_codes, b_scales, b_amax, K, rows, cols):
    """Sampled fp64 outputs of A (row-scaled NVFP4) x B^T (NVFP4, tensor amax b_amax)."""
    ga = np.array([nvfp4_g(float(v)) for v in np.asarray(a_amax_rows, np.float32)], np.float32)
    ac = np.ascontiguousarray(a_codes, dtype=np.uint8)
    asc = np.ascontiguousarray(a_scales, dtype=np.uint8)
    bc = np.ascontiguousarray(b_codes, dtype=np.uint8)
    bsc = np.ascontiguousarray(b_scales, dtype=np.uint8)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.zeros(r.size, np.float64)
    _load().orc_gemm_tn_sampled_rowscaled(_p(ac), _p(asc), _p(ga), _p(bc), _p(bsc), float(nvfp4_g(b_amax)), K,
                                          r.size, _p(r), _p(c), _p(out))
    return out


# ---------------------------------------------------------------- NVFP4 2D (16 x 16) columnwise scaling
def nvfp4_quantize_cols_2d(x, A: float | None = None):
    """Columnwise NVFP4 of bf16 x[M,K] with one scale per 16 x 16 tile ->
    (codes u8[K, Mp/2], compact scales u8[K, Mp/16], A); K % 16 == 0."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if A is None:
        A = amax(xb)
    nb = (M + 15) // 16
    codes = np.zeros((K, nb * 8), np.uint8)
    scales = np.zeros((K, nb), np.uint8)
    _load().orc_nvfp4_quantize_cols_2d(_p(xb), M, K, K, A, _p(codes), _p(scales))
    return codes, scales, A
