"""Block-scaled NVFP4 / MXFP8 quantization and GEMMs for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libnvq.so`` (declared in
``include/nvq.h``): argument marshalling only.  Every step of the path runs in
the library's CUDA kernels; PyTorch provides device memory and the current
stream.  Importing works without a GPU; any call that needs the library
raises if ``libnvq.so`` has not been built (there is no fallback).

Method pages: "Add an NVFP4 quantization converter" (torchtitan PR #3914) and
"Hybrid quantization" (TransformerEngine PR #2817).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

__all__ = [
    "NVFP4", "MXFP8", "IDENTITY", "NVFP4_ROWSCALED", "X_ROW_SCALED", "COL_2D", "W_COL_2D", "NONE",
    "hybrid_linear_fwd", "hybrid_linear_bwd_quantize", "linear_dgrad", "linear_wgrad", "DIR_ROW", "DIR_COL", "AMAX_GIVEN", "COL_SOURCE_ORIGINAL",
    "COL_SOURCE_ROWWISE_DEQUANTIZED", "NvqError", "QTensor", "lib", "load",
    "alloc_qtensor", "query_sizes", "colwise_cols", "amax", "nvfp4_quantize", "mxfp8_quantize",
    "hybrid_quantize", "gemm_tn", "nvfp4_linear_fwd", "nvfp4_linear_bwd_quantize",
    "nvfp4_linear_dgrad", "nvfp4_linear_wgrad", "grouped_padded_rows", "grouped_hybrid_quantize",
    "grouped_gemm_rows", "grouped_gemm_wgrad", "grouped_linear_fwd", "grouped_linear_bwd_quantize",
    "grouped_linear_dgrad", "grouped_linear_wgrad", "device_status", "gemm_pair_available",
    "EXPORTED_SYMBOLS",
]

NONE, NVFP4, MXFP8, IDENTITY, NVFP4_ROWSCALED = 0, 1, 2, 3, 4
X_ROW_SCALED = 2
COL_2D = 4
W_COL_2D = 4
COL_SOURCE_ORIGINAL, COL_SOURCE_ROWWISE_DEQUANTIZED = 0, 1
DIR_ROW, DIR_COL = 1, 2
AMAX_GIVEN = 1
MAX_GROUPS = 256

STATUS_NAMES = {0: "NVQ_OK", 1: "NVQ_ERR_NULL", 2: "NVQ_ERR_SHAPE", 3: "NVQ_ERR_ALIGN",
                4: "NVQ_ERR_WORKSPACE", 5: "NVQ_ERR_UNSUPPORTED", 6: "NVQ_ERR_CUDA",
                7: "NVQ_ERR_TIMEOUT", 8: "NVQ_ERR_BOUNDS"}


class NvqError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


class _QT(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("data", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class _SR(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_int64), ("offset", ctypes.c_uint32)]


class _RHT(ctypes.Structure):
    _fields_ = [("sign", ctypes.c_int8 * 16)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_QTP = ctypes.POINTER(_QT)
_SIGS = {
    "nvq_query_sizes": (_I32, [_I32, _I64, _I64, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "nvq_colwise_cols": (_I64, [_I32, _I64]),
    "nvq_amax": (_I32, [_P, _I64, _I64, _I64, ctypes.POINTER(_RHT), _P, _P, _P]),
    "nvq_nvfp4_quantize": (_I32, [_P, _I64, _I64, _I64, _I32, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _QTP, _QTP, _P]),
    "nvq_nvfp4_quantize_ex": (_I32, [_P, _I64, _I64, _I64, _I32, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _I32, _QTP, _QTP, _P]),
    "nvq_mxfp8_quantize": (_I32, [_P, _I64, _I64, _I64, _I32, _QTP, _QTP, _P]),
    "nvq_hybrid_quantize": (_I32, [_P, _I64, _I64, _I64, _I32, _I32, _I32, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _QTP, _QTP, _P]),
    "nvq_hybrid_quantize_ex": (_I32, [_P, _I64, _I64, _I64, _I32, _I32, _I32, ctypes.POINTER(_RHT), ctypes.POINTER(_SR),
                                      _I32, _QTP, _QTP, _P]),
    "nvq_hybrid_linear_fwd": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I32, _I32, ctypes.POINTER(_RHT), _I32, _P, _QTP,
                                     _QTP, _QTP, _QTP, _P]),
    "nvq_hybrid_linear_bwd_quantize": (_I32, [_P, _I64, _I64, _I32, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _QTP,
                                              _QTP, _P]),
    "nvq_linear_dgrad": (_I32, [_QTP, _QTP, _P, _P]),
    "nvq_linear_wgrad": (_I32, [_QTP, _QTP, _P, _P]),
    "nvq_gemm_tn": (_I32, [_QTP, _QTP, _P, _P, _I64, _I32, _P]),
    "nvq_gemm_tn_amax": (_I32, [_QTP, _QTP, _P, _P, _I64, _I32, ctypes.POINTER(_RHT), _P, _P, _P]),
    "nvq_nvfp4_linear_fwd": (_I32, [_P, _P, _P, _I64, _I64, _I64, ctypes.POINTER(_RHT), _P, _QTP, _QTP, _QTP, _QTP, _P]),
    "nvq_nvfp4_linear_fwd_ex": (_I32, [_P, _P, _P, _I64, _I64, _I64, ctypes.POINTER(_RHT), _I32, _P, _P, _P, _QTP, _QTP,
                                       _QTP, _QTP, _P]),
    "nvq_nvfp4_linear_bwd_quantize": (_I32, [_P, _I64, _I64, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _QTP, _QTP, _P]),
    "nvq_nvfp4_linear_bwd_quantize_ex": (_I32, [_P, _I64, _I64, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _I32, _QTP,
                                                _QTP, _P]),
    "nvq_nvfp4_linear_dgrad": (_I32, [_QTP, _QTP, _P, _P]),
    "nvq_nvfp4_linear_dgrad_ex": (_I32, [_QTP, _QTP, ctypes.POINTER(_RHT), _P, _P, _P, _P]),
    "nvq_nvfp4_linear_wgrad": (_I32, [_QTP, _QTP, _P, _P]),
    "nvq_grouped_padded_rows": (_I64, [ctypes.POINTER(_I64), _I32]),
    "nvq_grouped_hybrid_quantize": (_I32, [_P, _I64, _I64, ctypes.POINTER(_I64), _I32, _I32, _I32, _QTP, _QTP, ctypes.POINTER(_RHT), ctypes.POINTER(_SR), _P]),
    "nvq_grouped_gemm_rows": (_I32, [_QTP, _QTP, ctypes.POINTER(_I64), _I32, _I64, _I32, _P, _I64, _P]),
    "nvq_grouped_gemm_wgrad": (_I32, [_QTP, _QTP, ctypes.POINTER(_I64), _I32, _P, _I64, _P]),
    "nvq_grouped_linear_fwd": (_I32, [_P, _P, ctypes.POINTER(_I64), _I32, _I64, _I64, _P, _QTP, _QTP, _QTP, _QTP, _P]),
    "nvq_grouped_linear_fwd_ex": (_I32, [_P, _P, ctypes.POINTER(_I64), _I32, _I64, _I64, _I32, _P, _QTP, _QTP, _QTP,
                                         _QTP, _P]),
    "nvq_grouped_linear_bwd_quantize": (_I32, [_P, ctypes.POINTER(_I64), _I32, _I64, _QTP, _QTP, _P]),
    "nvq_grouped_linear_dgrad": (_I32, [_QTP, _QTP, ctypes.POINTER(_I64), _I32, _P, _P]),
    "nvq_grouped_linear_wgrad": (_I32, [_QTP, _QTP, ctypes.POINTER(_I64), _I32, _P, _P]),
    "nvq_status_string": (ctypes.c_char_p, [_I32]),
    "nvq_get_device_status": (_I32, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "nvq_gemm_pair_available": (_I32, []),
    "nvq_version": (ctypes.c_char_p, []),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libnvq.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"libnvq.so not built ({p}); run __graft_entry__.build()")
            L = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def lib():
    return load()


def _check(code: int, where: str):
    if code != 0:
        raise NvqError(code, where)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@dataclass
class QTensor:
    """A quantized K-major operand: ``rows`` rows of ``cols`` contraction
    elements; ``data`` codes, ``scale`` swizzled block scales, ``amax`` the
    per-tensor (or per-group) FP32 amax for NVFP4."""
    fmt: int
    rows: int
    cols: int
    data: torch.Tensor
    scale: torch.Tensor
    amax: Optional[torch.Tensor]

    def c(self) -> _QT:
        return _QT(self.fmt, self.data.data_ptr(), self.scale.data_ptr() if self.scale is not None else None,
                   self.amax.data_ptr() if self.amax is not None else None, self.rows, self.cols)

    def bf16(self) -> torch.Tensor:
        """The values of an IDENTITY operand as a bf16 [rows, cols] view."""
        if self.fmt != IDENTITY:
            raise ValueError("only an IDENTITY operand holds bf16 values")
        return self.data[: self.rows * self.cols * 2].view(torch.bfloat16).view(self.rows, self.cols)


def query_sizes(fmt: int, rows: int, cols: int):
    db, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().nvq_query_sizes(fmt, rows, cols, ctypes.byref(db), ctypes.byref(sb)), "nvq_query_sizes")
    return db.value, sb.value


def colwise_cols(fmt: int, M: int) -> int:
    return load().nvq_colwise_cols(fmt, M)


def alloc_qtensor(fmt: int, rows: int, cols: int, n_amax: Optional[int] = None, device="cuda") -> QTensor:
    """Storage for a [rows, cols] operand of `fmt`.  NVFP4 gets n_amax amaxes
    (default 1; one per group for grouped storage), row-scaled NVFP4 one per row."""
    db, sb = query_sizes(fmt, rows, cols)
    data = torch.empty(max(db, 16), dtype=torch.uint8, device=device)
    scale = torch.empty(max(sb, 16), dtype=torch.uint8, device=device) if fmt != IDENTITY else None
    if n_amax is None:
        n_amax = rows if fmt == NVFP4_ROWSCALED else 1
    amax = (torch.empty(max(n_amax, 1), dtype=torch.float32, device=device)
            if fmt in (NVFP4, NVFP4_ROWSCALED) else None)
    return QTensor(fmt, rows, cols, data, scale, amax)


def _sr(sr):
    if sr is None:
        return None
    seed, offset = (sr, 0) if isinstance(sr, int) else sr
    return ctypes.byref(_SR(int(seed), int(offset)))


def _rht(sign):
    if sign is None:
        return None
    vals = [int(v) for v in list(sign)]
    if len(vals) != 16:
        raise ValueError("RHT sign vector needs 16 entries")
    return ctypes.byref(_RHT((ctypes.c_int8 * 16)(*vals)))


def _bf16_2d(x: torch.Tensor):
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda:
        raise ValueError("expected a 2-D bf16 CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("innermost dimension must be contiguous")
    return x.shape[0], x.shape[1], x.stride(0)


def amax(x: torch.Tensor, rht_sign=None, stream=None):
    M, K, ld = _bf16_2d(x)
    a = torch.empty(1, dtype=torch.float32, device=x.device)
    r = torch.empty(1, dtype=torch.float32, device=x.device) if rht_sign is not None else None
    _check(load().nvq_amax(_ptr(x), M, K, ld, _rht(rht_sign), _ptr(a), _ptr(r), _stream(stream)), "nvq_amax")
    return a, r


def hybrid_quantize(x: torch.Tensor, row_fmt: int, col_fmt: int, rht_sign=None, sr=None, stream=None,
                    out_row: Optional[QTensor] = None, out_col: Optional[QTensor] = None,
                    col_source: int = COL_SOURCE_ORIGINAL, col_2d: bool = False):
    """Rowwise in ``row_fmt`` and columnwise in ``col_fmt`` (NVFP4, MXFP8 or
    IDENTITY); the columnwise source is the original x or, with
    COL_SOURCE_ROWWISE_DEQUANTIZED, the dequantized rowwise value."""
    M, K, ld = _bf16_2d(x)
    row = out_row or (alloc_qtensor(row_fmt, M, K, device=x.device) if row_fmt else None)
    col = out_col or (alloc_qtensor(col_fmt, K, colwise_cols(col_fmt, M), device=x.device) if col_fmt else None)
    rc, cc = (row.c() if row else None), (col.c() if col else None)
    _check(load().nvq_hybrid_quantize_ex(_ptr(x), M, K, ld, row_fmt, col_fmt, col_source, _rht(rht_sign), _sr(sr),
                                         COL_2D if col_2d else 0, ctypes.byref(rc) if rc else None,
                                         ctypes.byref(cc) if cc else None, _stream(stream)), "nvq_hybrid_quantize_ex")
    return row, col


def nvfp4_quantize(x: torch.Tensor, dirs: int = DIR_ROW | DIR_COL, rht_sign=None, sr=None, stream=None,
                   out_row: Optional[QTensor] = None, out_col: Optional[QTensor] = None, amax_given: bool = False,
                   col_2d: bool = False):
    """NVFP4 row and/or column quantization.  amax_given: the outputs' amax
    buffers already hold x's amaxes (written by the GEMM that produced x), so
    the amax pass is skipped."""
    M, K, ld = _bf16_2d(x)
    row = out_row or (alloc_qtensor(NVFP4, M, K, device=x.device) if dirs & DIR_ROW else None)
    col = out_col or (alloc_qtensor(NVFP4, K, colwise_cols(NVFP4, M), device=x.device) if dirs & DIR_COL else None)
    rc, cc = (row.c() if row else None), (col.c() if col else None)
    flags = (AMAX_GIVEN if amax_given else 0) | (COL_2D if col_2d else 0)
    _check(load().nvq_nvfp4_quantize_ex(_ptr(x), M, K, ld, dirs, _rht(rht_sign), _sr(sr), flags,
                                        ctypes.byref(rc) if rc else None, ctypes.byref(cc) if cc else None,
                                        _stream(stream)), "nvq_nvfp4_quantize_ex")
    return row, col


def mxfp8_quantize(x: torch.Tensor, dirs: int = DIR_ROW | DIR_COL, stream=None,
                   out_row: Optional[QTensor] = None, out_col: Optional[QTensor] = None):
    M, K, ld = _bf16_2d(x)
    row = out_row or (alloc_qtensor(MXFP8, M, K, device=x.device) if dirs & DIR_ROW else None)
    col = out_col or (alloc_qtensor(MXFP8, K, colwise_cols(MXFP8, M), device=x.device) if dirs & DIR_COL else None)
    rc, cc = (row.c() if row else None), (col.c() if col else None)
    _check(load().nvq_mxfp8_quantize(_ptr(x), M, K, ld, dirs, ctypes.byref(rc) if rc else None,
                                     ctypes.byref(cc) if cc else None, _stream(stream)), "nvq_mxfp8_quantize")
    return row, col


def gemm_tn(A: QTensor, B: QTensor, bias: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
            out: Optional[torch.Tensor] = None, stream=None, rht_sign=None, amax_out: Optional[torch.Tensor] = None,
            amax_rht_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """C[r, c] = alpha * sum_k A[r, k] B[c, k] (+ bias[c]).  amax_out /
    amax_rht_out (fp32 device tensors, element 0 written): the plain and
    Hadamard-domain (sign vector rht_sign) amaxes of the stored C."""
    if out is None:
        out = torch.empty(A.rows, B.rows, dtype=out_dtype, device=A.data.device)
    ac, bc = A.c(), B.c()
    c32 = 1 if out.dtype == torch.float32 else 0
    if amax_out is None and amax_rht_out is None:
        _check(load().nvq_gemm_tn(ctypes.byref(ac), ctypes.byref(bc), _ptr(bias), _ptr(out), out.stride(0), c32,
                                  _stream(stream)), "nvq_gemm_tn")
    else:
        _check(load().nvq_gemm_tn_amax(ctypes.byref(ac), ctypes.byref(bc), _ptr(bias), _ptr(out), out.stride(0), c32,
                                       _rht(rht_sign), _ptr(amax_out), _ptr(amax_rht_out), _stream(stream)),
               "nvq_gemm_tn_amax")
    return out


def nvfp4_linear_fwd(x: torch.Tensor, w: torch.Tensor, bias=None, rht_sign=None, save_for_backward=True,
                     stream=None, y: Optional[torch.Tensor] = None, bufs=None, amax_given: bool = False,
                     y_amax: Optional[torch.Tensor] = None, y_amax_rht: Optional[torch.Tensor] = None):
    """y = x W^T with NVFP4 operands; returns (y, saved) where saved holds the
    quantized x_row, w_row, the RHT'd columnwise x (wgrad) and columnwise W (dgrad).
    amax_given: bufs["x_row"].amax / bufs["x_col"].amax already hold x's
    amaxes; y_amax / y_amax_rht receive y's amaxes for the next layer."""
    M, K, _ = _bf16_2d(x)
    N = w.shape[0]
    if bufs is None:
        bufs = dict(x_row=alloc_qtensor(NVFP4, M, K, device=x.device),
                    w_row=alloc_qtensor(NVFP4, N, K, device=x.device),
                    x_col=alloc_qtensor(NVFP4, K, colwise_cols(NVFP4, M), device=x.device) if save_for_backward else None,
                    w_col=alloc_qtensor(NVFP4, K, colwise_cols(NVFP4, N), device=x.device) if save_for_backward else None)
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    xr, wr = bufs["x_row"].c(), bufs["w_row"].c()
    xc = bufs["x_col"].c() if bufs.get("x_col") is not None else _QT()
    wc = bufs["w_col"].c() if bufs.get("w_col") is not None else _QT()
    _check(load().nvq_nvfp4_linear_fwd_ex(_ptr(x), _ptr(w), _ptr(bias), M, N, K, _rht(rht_sign),
                                          AMAX_GIVEN if amax_given else 0, _ptr(y), _ptr(y_amax), _ptr(y_amax_rht),
                                          ctypes.byref(xr), ctypes.byref(wr), ctypes.byref(xc), ctypes.byref(wc),
                                          _stream(stream)), "nvq_nvfp4_linear_fwd_ex")
    return y, bufs


def nvfp4_linear_bwd_quantize(dy: torch.Tensor, rht_sign=None, sr=None, stream=None, bufs=None,
                              amax_given: bool = False):
    M, N, _ = _bf16_2d(dy)
    if bufs is None:
        bufs = dict(dy_row=alloc_qtensor(NVFP4, M, N, device=dy.device),
                    dy_col=alloc_qtensor(NVFP4, N, colwise_cols(NVFP4, M), device=dy.device))
    r, c = bufs["dy_row"].c(), bufs["dy_col"].c()
    _check(load().nvq_nvfp4_linear_bwd_quantize_ex(_ptr(dy), M, N, _rht(rht_sign), _sr(sr),
                                                   AMAX_GIVEN if amax_given else 0, ctypes.byref(r), ctypes.byref(c),
                                                   _stream(stream)), "nvq_nvfp4_linear_bwd_quantize_ex")
    return bufs


def nvfp4_linear_dgrad(dy_row: QTensor, w_col: QTensor, dx: Optional[torch.Tensor] = None, stream=None,
                       rht_sign=None, dx_amax: Optional[torch.Tensor] = None,
                       dx_amax_rht: Optional[torch.Tensor] = None):
    if dx is None:
        dx = torch.empty(dy_row.rows, w_col.rows, dtype=torch.bfloat16, device=dy_row.data.device)
    a, b = dy_row.c(), w_col.c()
    _check(load().nvq_nvfp4_linear_dgrad_ex(ctypes.byref(a), ctypes.byref(b), _rht(rht_sign), _ptr(dx), _ptr(dx_amax),
                                            _ptr(dx_amax_rht), _stream(stream)), "nvq_nvfp4_linear_dgrad_ex")
    return dx


def nvfp4_linear_wgrad(dy_col: QTensor, x_col: QTensor, dw: Optional[torch.Tensor] = None, stream=None):
    if dw is None:
        dw = torch.empty(dy_col.rows, x_col.rows, dtype=torch.bfloat16, device=dy_col.data.device)
    a, b = dy_col.c(), x_col.c()
    _check(load().nvq_nvfp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), _ptr(dw), _stream(stream)),
           "nvq_nvfp4_linear_wgrad")
    return dw


def hybrid_linear_fwd(x: torch.Tensor, w: torch.Tensor, fwd_fmt: int, bwd_fmt: int, bias=None, rht_sign=None,
                      w_col_2d: bool = False, save_for_backward=True, stream=None, y: Optional[torch.Tensor] = None,
                      bufs=None):
    """Linear forward with per-direction formats (e.g. MXFP8 forward, NVFP4
    backward): y = x W^T in fwd_fmt; saved x_col / w_col in bwd_fmt."""
    M, K, _ = _bf16_2d(x)
    N = w.shape[0]
    if bufs is None:
        bufs = dict(x_row=alloc_qtensor(fwd_fmt, M, K, device=x.device), w_row=alloc_qtensor(fwd_fmt, N, K, device=x.device),
                    x_col=alloc_qtensor(bwd_fmt, K, colwise_cols(bwd_fmt, M), device=x.device) if save_for_backward else None,
                    w_col=alloc_qtensor(bwd_fmt, K, colwise_cols(bwd_fmt, N), device=x.device) if save_for_backward else None)
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    xr, wr = bufs["x_row"].c(), bufs["w_row"].c()
    xc = bufs["x_col"].c() if bufs.get("x_col") is not None else _QT()
    wc = bufs["w_col"].c() if bufs.get("w_col") is not None else _QT()
    _check(load().nvq_hybrid_linear_fwd(_ptr(x), _ptr(w), _ptr(bias), M, N, K, fwd_fmt, bwd_fmt, _rht(rht_sign),
                                        W_COL_2D if w_col_2d else 0, _ptr(y), ctypes.byref(xr), ctypes.byref(wr),
                                        ctypes.byref(xc), ctypes.byref(wc), _stream(stream)), "nvq_hybrid_linear_fwd")
    return y, bufs


def hybrid_linear_bwd_quantize(dy: torch.Tensor, bwd_fmt: int, rht_sign=None, sr=None, stream=None, bufs=None):
    M, N, _ = _bf16_2d(dy)
    if bufs is None:
        bufs = dict(dy_row=alloc_qtensor(bwd_fmt, M, N, device=dy.device),
                    dy_col=alloc_qtensor(bwd_fmt, N, colwise_cols(bwd_fmt, M), device=dy.device))
    r, c = bufs["dy_row"].c(), bufs["dy_col"].c()
    _check(load().nvq_hybrid_linear_bwd_quantize(_ptr(dy), M, N, bwd_fmt, _rht(rht_sign), _sr(sr), ctypes.byref(r),
                                                 ctypes.byref(c), _stream(stream)), "nvq_hybrid_linear_bwd_quantize")
    return bufs


def linear_dgrad(dy_row: QTensor, w_col: QTensor, dx: Optional[torch.Tensor] = None, stream=None):
    if dx is None:
        dx = torch.empty(dy_row.rows, w_col.rows, dtype=torch.bfloat16, device=dy_row.data.device)
    a, b = dy_row.c(), w_col.c()
    _check(load().nvq_linear_dgrad(ctypes.byref(a), ctypes.byref(b), _ptr(dx), _stream(stream)), "nvq_linear_dgrad")
    return dx


def linear_wgrad(dy_col: QTensor, x_col: QTensor, dw: Optional[torch.Tensor] = None, stream=None):
    if dw is None:
        dw = torch.empty(dy_col.rows, x_col.rows, dtype=torch.bfloat16, device=dy_col.data.device)
    a, b = dy_col.c(), x_col.c()
    _check(load().nvq_linear_wgrad(ctypes.byref(a), ctypes.byref(b), _ptr(dw), _stream(stream)), "nvq_linear_wgrad")
    return dw


def _groups(group_rows: Sequence[int]):
    g = [int(v) for v in group_rows]
    return (_I64 * len(g))(*g), len(g)


def grouped_padded_rows(group_rows: Sequence[int]) -> int:
    arr, G = _groups(group_rows)
    return load().nvq_grouped_padded_rows(arr, G)


def grouped_hybrid_quantize(x: torch.Tensor, group_rows: Sequence[int], row_fmt: int, col_fmt: int,
                            stream=None, out_row: Optional[QTensor] = None, out_col: Optional[QTensor] = None,
                            rht_sign=None, sr=None):
    """Per-group hybrid quantization; storage padded to 128 rows per group.
    rht_sign / sr: RHT on an NVFP4 columnwise direction, SR on NVFP4
    directions (stochastic-rounding index = position in the padded output)."""
    M, K, ld = _bf16_2d(x)
    arr, G = _groups(group_rows)
    P = load().nvq_grouped_padded_rows(arr, G)
    row = out_row or (alloc_qtensor(row_fmt, P, K, n_amax=P if row_fmt == NVFP4_ROWSCALED else G, device=x.device)
                      if row_fmt else None)
    col = out_col or (alloc_qtensor(col_fmt, K, P, n_amax=G, device=x.device) if col_fmt else None)
    rc, cc = (row.c() if row else None), (col.c() if col else None)
    _check(load().nvq_grouped_hybrid_quantize(_ptr(x), K, ld, arr, G, row_fmt, col_fmt,
                                              ctypes.byref(rc) if rc else None, ctypes.byref(cc) if cc else None,
                                              _rht(rht_sign), _sr(sr), _stream(stream)), "nvq_grouped_hybrid_quantize")
    return row, col


def grouped_gemm_rows(A: QTensor, B: QTensor, group_rows: Sequence[int], n_per_group: int, b_col_groups: bool,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    arr, G = _groups(group_rows)
    n_out = n_per_group if not b_col_groups else B.rows
    if out is None:
        out = torch.empty(sum(int(v) for v in group_rows), n_out, dtype=torch.bfloat16, device=A.data.device)
    ac, bc = A.c(), B.c()
    _check(load().nvq_grouped_gemm_rows(ctypes.byref(ac), ctypes.byref(bc), arr, G, n_per_group,
                                        1 if b_col_groups else 0, _ptr(out), out.stride(0), _stream(stream)),
           "nvq_grouped_gemm_rows")
    return out


def grouped_gemm_wgrad(A: QTensor, B: QTensor, group_rows: Sequence[int], out: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    arr, G = _groups(group_rows)
    if out is None:
        out = torch.empty(G, A.rows, B.rows, dtype=torch.bfloat16, device=A.data.device)
    ac, bc = A.c(), B.c()
    _check(load().nvq_grouped_gemm_wgrad(ctypes.byref(ac), ctypes.byref(bc), arr, G, _ptr(out), out.stride(-2),
                                         _stream(stream)), "nvq_grouped_gemm_wgrad")
    return out


def grouped_linear_fwd(x: torch.Tensor, w: torch.Tensor, group_rows: Sequence[int], stream=None,
                       y: Optional[torch.Tensor] = None, bufs=None, save_for_backward=True, row_scaled_x: bool = False):
    """Grouped (MoE) linear forward, NVFP4: x [T][K], w [G][N][K] or [G*N][K];
    returns (y [T][N], bufs) with bufs holding x_row, w_row and, for the
    backward, MXFP8 x_col and w_col.  row_scaled_x: x's rowwise direction is
    row-scaled NVFP4 (one FP32 outer scale per row)."""
    T, K, _ = _bf16_2d(x)
    arr, G = _groups(group_rows)
    w2 = w.reshape(-1, w.shape[-1])
    N = w2.shape[0] // G
    P = load().nvq_grouped_padded_rows(arr, G)
    if bufs is None:
        bufs = dict(x_row=(alloc_qtensor(NVFP4_ROWSCALED, P, K, device=x.device) if row_scaled_x
                           else alloc_qtensor(NVFP4, P, K, n_amax=G, device=x.device)),
                    w_row=alloc_qtensor(NVFP4, G * N, K, n_amax=G, device=x.device),
                    x_col=alloc_qtensor(MXFP8, K, P, device=x.device) if save_for_backward else None,
                    w_col=alloc_qtensor(MXFP8, K, G * N, device=x.device) if save_for_backward else None)
    if y is None:
        y = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    xr, wr = bufs["x_row"].c(), bufs["w_row"].c()
    xc = bufs["x_col"].c() if bufs.get("x_col") is not None else _QT()
    wc = bufs["w_col"].c() if bufs.get("w_col") is not None else _QT()
    _check(load().nvq_grouped_linear_fwd_ex(_ptr(x), _ptr(w2), arr, G, N, K, X_ROW_SCALED if row_scaled_x else 0,
                                            _ptr(y), ctypes.byref(xr), ctypes.byref(wr), ctypes.byref(xc),
                                            ctypes.byref(wc), _stream(stream)), "nvq_grouped_linear_fwd_ex")
    return y, bufs


def grouped_linear_bwd_quantize(dy: torch.Tensor, group_rows: Sequence[int], stream=None, bufs=None):
    """dy [T][N] -> MXFP8 dy_row [P][N] and dy_col [N][P] (grouped)."""
    T, N, _ = _bf16_2d(dy)
    arr, G = _groups(group_rows)
    P = load().nvq_grouped_padded_rows(arr, G)
    if bufs is None:
        bufs = dict(dy_row=alloc_qtensor(MXFP8, P, N, device=dy.device), dy_col=alloc_qtensor(MXFP8, N, P, device=dy.device))
    r, c = bufs["dy_row"].c(), bufs["dy_col"].c()
    _check(load().nvq_grouped_linear_bwd_quantize(_ptr(dy), arr, G, N, ctypes.byref(r), ctypes.byref(c), _stream(stream)),
           "nvq_grouped_linear_bwd_quantize")
    return bufs


def grouped_linear_dgrad(dy_row: QTensor, w_col: QTensor, group_rows: Sequence[int],
                         dx: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    arr, G = _groups(group_rows)
    if dx is None:
        dx = torch.empty(sum(int(v) for v in group_rows), w_col.rows, dtype=torch.bfloat16, device=dy_row.data.device)
    a, b = dy_row.c(), w_col.c()
    _check(load().nvq_grouped_linear_dgrad(ctypes.byref(a), ctypes.byref(b), arr, G, _ptr(dx), _stream(stream)),
           "nvq_grouped_linear_dgrad")
    return dx


def grouped_linear_wgrad(dy_col: QTensor, x_col: QTensor, group_rows: Sequence[int],
                         dw: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    arr, G = _groups(group_rows)
    if dw is None:
        dw = torch.empty(G, dy_col.rows, x_col.rows, dtype=torch.bfloat16, device=dy_col.data.device)
    a, b = dy_col.c(), x_col.c()
    _check(load().nvq_grouped_linear_wgrad(ctypes.byref(a), ctypes.byref(b), arr, G, _ptr(dw), _stream(stream)),
           "nvq_grouped_linear_wgrad")
    return dw


def gemm_pair_available() -> bool:
    """True when GEMMs with an output width divisible by 256 run on the CTA-pair kernel."""
    v = load().nvq_gemm_pair_available()
    if v < 0:
        raise NvqError(6, "nvq_gemm_pair_available")
    return v == 1


def device_status(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().nvq_get_device_status(_stream(stream), ctypes.byref(code)), "nvq_get_device_status")
    return code.value
