"""CPU oracle for the quantized lightning indexer — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this package. It wraps the plain C statement of the indexer in
``qli_oracle.c`` (which cites the page passages it follows) and shares no code
with the CUDA library. Inputs are host numpy arrays; any object carrying the
attributes of a batch (q, cu_seqlens_q, k_lens, ...) can be passed.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_lib = None


class _In(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_stride_t", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
        ("T", ctypes.c_int32), ("N", ctypes.c_int32), ("D", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("B", ctypes.c_int32),
        ("k_lens", ctypes.c_void_p), ("residual", ctypes.c_void_p),
        ("cache", ctypes.c_void_p), ("page_stride", ctypes.c_int64),
        ("rows_per_page", ctypes.c_int32),
        ("k_offset", ctypes.c_int64), ("scale_offset", ctypes.c_int64),
        ("num_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
        ("head_weights", ctypes.c_void_p), ("q_scale", ctypes.c_void_p),
        ("ratio", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("cand_mode", ctypes.c_int32), ("cand_blocks", ctypes.c_int32),
        ("cand_in", ctypes.c_void_p),
        ("quant_mode", ctypes.c_int32),
    ]


ERRORS = {-1: "invalid argument", -3: "consumer without source", -4: "residual with ratio 1"}
MODES = {"none": 1, "source": 2, "consumer": 3}


class OracleError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB points the wrapper at another build of qli_oracle.c (the
        # mutation tests use it to check that the pins catch planted mistakes)
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.oracle_qli.restype = ctypes.c_int
        L.oracle_qli.argtypes = [ctypes.POINTER(_In), ctypes.c_void_p, ctypes.c_int32,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32]
        L.oracle_visible_count.restype = ctypes.c_int64
        L.oracle_visible_count.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                           ctypes.c_int64, ctypes.c_int64]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_head_term.restype = ctypes.c_float
        L.oracle_head_term.argtypes = [ctypes.c_int32, ctypes.c_uint16, ctypes.c_uint16]
        L.oracle_dot.restype = ctypes.c_int32
        L.oracle_dot.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        L.oracle_pair_score.restype = ctypes.c_float
        L.oracle_pair_score.argtypes = [ctypes.POINTER(_In), ctypes.c_int32, ctypes.c_int64]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_dot_e4m3.restype = ctypes.c_float
        L.oracle_dot_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        L.oracle_head_term_f8.restype = ctypes.c_float
        L.oracle_head_term_f8.argtypes = [ctypes.c_float, ctypes.c_uint16, ctypes.c_uint16]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class Prepared:
    """Holds the C argument struct and keeps its arrays alive."""

    def __init__(self, case, pages: np.ndarray, page_stride: int, k_offset: int,
                 scale_offset: int, cand_mode: Optional[str] = None,
                 cand_in: Optional[np.ndarray] = "from_case", residual="from_case"):
        mode = case.cand_mode if cand_mode is None else cand_mode
        self.keep = []

        def c(a, dt):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=dt)
            self.keep.append(a)
            return a

        # FP8 cases carry E4M3 bit patterns: the bytes are passed unchanged
        q = c(np.asarray(case.q).view(np.int8) if np.asarray(case.q).dtype == np.uint8 else case.q,
              np.int8)
        T, N, D = q.shape
        pages = np.ascontiguousarray(pages)
        self.keep.append(pages)
        res = case.residual if isinstance(residual, str) else residual
        cin = case.cand_in if isinstance(cand_in, str) else cand_in
        s = _In()
        s.q = _ptr(q); s.q_stride_t = N * D; s.q_stride_h = D
        s.T, s.N, s.D = T, N, D
        s.cu_seqlens_q = _ptr(c(case.cu_seqlens_q, np.int32)); s.B = len(case.k_lens)
        s.k_lens = _ptr(c(case.k_lens, np.int32)); s.residual = _ptr(c(res, np.int32))
        s.cache = _ptr(pages); s.page_stride = page_stride
        s.rows_per_page = case.rows_per_page
        s.k_offset = k_offset; s.scale_offset = scale_offset
        s.num_pages = pages.shape[0]
        bt = c(case.block_table, np.int32)
        s.block_table = _ptr(bt); s.bt_stride = bt.shape[1]
        s.head_weights = _ptr(c(case.head_weights, np.uint16))
        s.q_scale = _ptr(c(case.q_scale, np.uint16))
        s.ratio = case.ratio; s.topk = case.topk
        s.cand_mode = MODES[mode]; s.cand_blocks = case.cand_blocks
        s.cand_in = _ptr(c(cin, np.int32))
        s.quant_mode = int(getattr(case, "quant_mode", 2))
        self.s = s
        self.T = T
        self.topk = case.topk
        self.cand_blocks = case.cand_blocks
        self.mode = mode


def prepare(case, pages: Optional[np.ndarray] = None, compact: bool = True, **kw) -> Prepared:
    """Packs the case's paged cache on the host (compact geometry by default:
    stride R*130, index K at offset 0, scales at R*128) and builds the struct."""
    if pages is None:
        if compact:
            R = case.rows_per_page
            stride, ko, so = R * 130, 0, R * 128
        else:
            stride, ko, so = case.page_stride, case.k_offset, case.scale_offset
        pages = case.pack_pages_numpy(page_stride=stride, k_offset=ko, scale_offset=so,
                                      filler=not compact)
        return Prepared(case, pages, stride, ko, so, **kw)
    return Prepared(case, pages, case.page_stride, case.k_offset, case.scale_offset, **kw)


def run(prep: Prepared, rows: Optional[Sequence[int]] = None, want_scores: bool = False,
        score_stride: Optional[int] = None, nthreads: int = 0):
    """Runs the oracle on the listed query tokens (all by default).

    Returns dict(indices [n, K], cand [n, C] or None, visible [n],
    scores [n, score_stride] float32 (NaN where j >= V) or None).
    """
    L = lib()
    rows = np.arange(prep.T, dtype=np.int32) if rows is None else np.asarray(rows, dtype=np.int32)
    n = rows.size
    idx = np.empty((n, prep.topk), dtype=np.int32)
    cand = (np.empty((n, prep.cand_blocks), dtype=np.int32)
            if prep.mode == "source" else None)
    vis = np.empty(n, dtype=np.int64)
    scores = None
    if want_scores:
        if score_stride is None:
            R = prep.s.rows_per_page
            score_stride = prep.s.bt_stride * R
        scores = np.full((n, score_stride), np.nan, dtype=np.float32)
    rc = L.oracle_qli(ctypes.byref(prep.s), _ptr(rows), n, _ptr(idx), _ptr(cand),
                      _ptr(scores), 0 if scores is None else score_stride, _ptr(vis), nthreads)
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))
    return {"indices": idx, "cand": cand, "visible": vis, "scores": scores}


def visible_count(k_len: int, residual: int, ratio: int, q_len: int, i: int) -> int:
    return int(lib().oracle_visible_count(k_len, residual, ratio, q_len, i))


def f32_to_f16_bits(x: float) -> int:
    return int(lib().oracle_f32_to_f16(float(x)))


def f16_bits_to_f32(b: int) -> float:
    return float(lib().oracle_f16_to_f32(int(b)))


def head_term(s: int, w_bits: int, qs_bits: int) -> float:
    return float(lib().oracle_head_term(int(s), int(w_bits), int(qs_bits)))


def pair_score(prep: Prepared, t: int, j: int) -> float:
    return float(lib().oracle_pair_score(ctypes.byref(prep.s), int(t), int(j)))


# ---- FP8 (quant mode 1): E4M3 codes ----------------------------------------

def e4m3_to_f64(code: int) -> float:
    return float(lib().oracle_e4m3_to_f64(int(code)))


def dot_e4m3(q_codes: np.ndarray, k_codes: np.ndarray) -> float:
    q = np.ascontiguousarray(q_codes, dtype=np.uint8)
    k = np.ascontiguousarray(k_codes, dtype=np.uint8)
    assert q.size == k.size
    return float(lib().oracle_dot_e4m3(_ptr(q), _ptr(k), q.size))


def head_term_f8(s: float, w_bits: int, qs_bits: int) -> float:
    return float(lib().oracle_head_term_f8(float(s), int(w_bits), int(qs_bits)))


# ---- query quantiser and index-K writer (qli_quant_oracle.c) ---------------

QUANT_ERRORS = {-1: "invalid argument", -2: "non-finite input", -5: "slot out of range"}


def _quant_fn(name, restype, argtypes):
    f = getattr(lib(), name)
    f.restype = restype
    f.argtypes = argtypes
    return f


def bf16_bits_to_f32(b: int) -> float:
    return float(_quant_fn("oracle_bf16_to_f32", ctypes.c_float, [ctypes.c_uint16])(int(b)))


def quantize_rows(x_bf16: np.ndarray):
    """Per-row INT8 quantisation of BF16 rows (given as uint16 bit patterns,
    shape [..., D]). Returns (codes int8 [..., D], scales uint16 [...] FP16 bits)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[-1]
    rows = x.size // D if D else 0
    q = np.empty(x.shape, dtype=np.int8)
    s = np.empty(x.shape[:-1], dtype=np.uint16)
    f = _quant_fn("oracle_quantize_rows", ctypes.c_int,
                  [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p])
    rc = f(_ptr(x), rows, D, _ptr(q), _ptr(s))
    if rc != 0:
        raise OracleError(QUANT_ERRORS.get(rc, str(rc)))
    return q, s


def quantize_rows_e4m3(x_bf16: np.ndarray):
    """FP8 variant: per-row E4M3 quantisation of BF16 rows (uint16 bit
    patterns, shape [..., D]). Returns (codes uint8 [..., D] E4M3 bits,
    scales uint16 [...] FP16 bits)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[-1]
    rows = x.size // D if D else 0
    c = np.empty(x.shape, dtype=np.uint8)
    s = np.empty(x.shape[:-1], dtype=np.uint16)
    f = _quant_fn("oracle_quantize_rows_e4m3", ctypes.c_int,
                  [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p])
    rc = f(_ptr(x), rows, D, _ptr(c), _ptr(s))
    if rc != 0:
        raise OracleError(QUANT_ERRORS.get(rc, str(rc)))
    return c, s


def f32_to_e4m3(x: float) -> int:
    return int(_quant_fn("oracle_f32_to_e4m3", ctypes.c_uint8, [ctypes.c_float])(float(x)))


def write_index_k(k_bf16: np.ndarray, slot: np.ndarray, pages: np.ndarray, rows_per_page: int,
                  k_offset: int, scale_offset: int, fp8: bool = False) -> int:
    """Quantises the n rows of k_bf16 ([n, D] uint16 BF16 bits; INT8 codes, or
    E4M3 codes when fp8) and writes them into `pages` ([num_pages,
    page_stride] uint8, modified in place) at slot[i] = page * R + row.
    Returns the oracle's status (0, or -5 when a slot lies past the pool;
    valid rows are written either way)."""
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    sl = np.ascontiguousarray(slot, dtype=np.int64)
    assert pages.flags.c_contiguous and pages.dtype == np.uint8 and pages.ndim == 2
    f = _quant_fn("oracle_write_index_k_e4m3" if fp8 else "oracle_write_index_k", ctypes.c_int,
                  [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                   ctypes.c_int64, ctypes.c_int64])
    rc = f(_ptr(k), k.shape[0], k.shape[1], _ptr(sl), _ptr(pages), pages.shape[0],
           pages.shape[1], rows_per_page, k_offset, scale_offset)
    if rc not in (0, -5):
        raise OracleError(QUANT_ERRORS.get(rc, str(rc)))
    return int(rc)
