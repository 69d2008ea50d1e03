"""Python binding of the C-ABI indexer library (include/qli.h).

Argument marshalling only: every step of the indexer runs in the library's
CUDA kernels. PyTorch supplies device memory and the stream. There is no
fallback: a missing library or a non-CUDA tensor raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_int32, c_int64, c_size_t, c_uint32, c_void_p
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libqli_gb300.so")

OK = 0
STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported", 3: "consumer without source",
    4: "residual with ratio 1", 5: "workspace too small", 6: "alignment", 7: "CUDA error",
    8: "not an sm_103 device",
}
CAND_MODES = {"none": 1, "source": 2, "consumer": 3}
STAGE_PLAN, STAGE_SCORE, STAGE_SELECT = 1, 2, 3
LAYOUT_TND, LAYOUT_PA_BBND, QUANT_INT8, MASK_CAUSAL = 1, 2, 2, 3
QUANT_FP8 = 1            # q and the index K hold E4M3 codes (passed as int8 bytes)
DEVERR = {1: "cu_seqlens", 2: "k_lens", 4: "residual", 8: "block table page", 16: "wait timeout"}


class QLIError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s" % (what or "qli", STATUS.get(status, str(status))))


class Args(ctypes.Structure):
    """Mirror of `qli_args` (field order and types as in include/qli.h)."""
    _fields_ = [
        ("q", c_void_p), ("q_stride_t", c_int64), ("q_stride_h", c_int64),
        ("T", c_int32), ("N", c_int32), ("D", c_int32),
        ("cu_seqlens_q", c_void_p), ("B", c_int32),
        ("k_lens", c_void_p), ("residual", c_void_p),
        ("cache", c_void_p), ("page_stride", c_int64), ("rows_per_page", c_int32),
        ("k_offset", c_int64), ("scale_offset", c_int64), ("num_pages", c_int64),
        ("block_table", c_void_p), ("bt_stride", c_int32),
        ("head_weights", c_void_p), ("q_scale", c_void_p),
        ("ratio", c_int32), ("mask_mode", c_int32), ("quant_mode", c_int32),
        ("layout_q", c_int32), ("layout_k", c_int32),
        ("topk", c_int32), ("cand_mode", c_int32), ("cand_blocks", c_int32),
        ("block_size", c_int32),
        ("cand_in", c_void_p), ("cand_in_numel", c_int64),
        ("cand_out", c_void_p), ("cand_out_numel", c_int64),
        ("indices_out", c_void_p), ("indices_numel", c_int64),
    ]


class AttnArgs(ctypes.Structure):
    """Mirror of `qli_attn_args` (field order and types as in include/qli.h)."""
    _fields_ = [
        ("q", c_void_p), ("q_stride_t", c_int64), ("q_stride_h", c_int64),
        ("T", c_int32), ("H", c_int32), ("D", c_int32),
        ("cu_seqlens_q", c_void_p), ("B", c_int32),
        ("cache", c_void_p), ("page_stride", c_int64), ("num_pages", c_int64),
        ("rows_per_page", c_int32), ("kv_offset", c_int64),
        ("block_table", c_void_p), ("bt_stride", c_int32),
        ("indices", c_void_p), ("K", c_int32), ("scale", ctypes.c_float),
        ("out", c_void_p), ("out_stride_t", c_int64), ("out_stride_h", c_int64),
        ("lse", c_void_p), ("err_word", c_void_p),
    ]


EXPORTS = ["qli_validate", "qli_workspace_size", "qli_run", "qli_run_stage", "qli_launch_count",
           "qli_scores_layout", "qli_read_device_error", "qli_status_string", "qli_abi_version",
           "qli_args_size", "qli_run_static", "qli_read_static_device_error",
           "qli_quantize_q", "qli_write_index_k", "qli_quantize_q_fp8", "qli_write_index_k_fp8",
           "qli_check_quant_rounding",
           "qli_sparse_attention", "qli_attn_args_size"]

_lib = None


def lib(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libqli_gb300.so (built by `build()`); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    # QLI_LIB selects another build of the same library (diagnostic variants)
    p = path or os.environ.get("QLI_LIB") or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libqli_gb300.so not built (run __graft_entry__.build() or "
                          "python -m sparse_attention_indexer_qli_gb300.build)")
    L = ctypes.CDLL(p)
    P = ctypes.POINTER(Args)
    L.qli_validate.argtypes = [P]
    L.qli_workspace_size.argtypes = [P, ctypes.POINTER(c_size_t)]
    L.qli_run.argtypes = [P, c_void_p, c_size_t, c_void_p]
    L.qli_run_stage.argtypes = [P, c_void_p, c_size_t, c_int32, c_void_p]
    L.qli_launch_count.argtypes = [P, c_int32, ctypes.POINTER(c_int32)]
    L.qli_scores_layout.argtypes = [P, ctypes.POINTER(c_size_t), ctypes.POINTER(c_int64)]
    L.qli_read_device_error.argtypes = [c_void_p, ctypes.POINTER(c_uint32), c_void_p]
    L.qli_run_static.argtypes = [P, c_void_p]
    L.qli_run_static.restype = c_int32
    L.qli_read_static_device_error.argtypes = [ctypes.POINTER(c_uint32), c_void_p]
    L.qli_read_static_device_error.restype = c_int32
    L.qli_status_string.argtypes = [c_int32]
    L.qli_status_string.restype = ctypes.c_char_p
    L.qli_abi_version.restype = c_int32
    L.qli_args_size.restype = c_int64
    for name in ("qli_quantize_q", "qli_quantize_q_fp8"):
        getattr(L, name).argtypes = [c_void_p, c_int64, c_void_p, c_void_p, c_void_p]
        getattr(L, name).restype = c_int32
    for name in ("qli_write_index_k", "qli_write_index_k_fp8"):
        getattr(L, name).argtypes = [c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_int64,
                                    c_int32, c_int64, c_int64, c_void_p, c_void_p]
        getattr(L, name).restype = c_int32
    L.qli_check_quant_rounding.argtypes = [c_void_p, c_void_p]
    L.qli_check_quant_rounding.restype = c_int32
    L.qli_sparse_attention.argtypes = [ctypes.POINTER(AttnArgs), c_void_p]
    L.qli_sparse_attention.restype = c_int32
    L.qli_attn_args_size.restype = c_int64
    if L.qli_attn_args_size() != ctypes.sizeof(AttnArgs):
        raise ImportError("qli_attn_args layout mismatch")
    for name in ["qli_validate", "qli_workspace_size", "qli_run", "qli_run_stage",
                 "qli_launch_count", "qli_scores_layout", "qli_read_device_error"]:
        getattr(L, name).restype = c_int32
    if L.qli_args_size() != ctypes.sizeof(Args):
        raise ImportError("qli_args layout mismatch: library %d bytes, binding %d bytes"
                          % (L.qli_args_size(), ctypes.sizeof(Args)))
    if path is None:
        _lib = L
    return L


def _check(st: int, what: str):
    if st != OK:
        raise QLIError(st, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _require_cuda(name, t, dtype=None):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


class Call:
    """One prepared indexer call: the argument struct plus the tensors it
    points into (kept alive here)."""

    def __init__(self, q, cu_seqlens_q, k_lens, residual, cache, block_table, head_weights,
                 q_scale, *, ratio: int, rows_per_page: int, page_stride: int, k_offset: int,
                 scale_offset: int, topk: int, cand_mode: str = "none", cand_blocks: int = 0,
                 cand_in=None, indices_out=None, cand_out=None, quant_mode: int = QUANT_INT8):
        import torch
        _require_cuda("q", q, torch.int8)
        for n, t in (("cu_seqlens_q", cu_seqlens_q), ("k_lens", k_lens), ("residual", residual),
                     ("block_table", block_table), ("cand_in", cand_in)):
            _require_cuda(n, t, torch.int32)
        _require_cuda("cache", cache, torch.uint8)
        _require_cuda("head_weights", head_weights, torch.float16)
        _require_cuda("q_scale", q_scale, torch.float16)
        if q.dim() != 3 or q.stride(2) != 1:
            raise ValueError("q must be [T, N, D] with unit stride in D")
        if block_table.dim() != 2 or block_table.stride(1) != 1:
            raise ValueError("block_table must be [B, bt_stride] row-major")
        for n, t in (("head_weights", head_weights), ("q_scale", q_scale)):
            if not t.is_contiguous():
                raise ValueError("%s must be contiguous [T, N]" % n)
        if not cache.is_contiguous():
            raise ValueError("cache must be contiguous")
        T, N, D = q.shape
        B = k_lens.numel()
        mode = CAND_MODES[cand_mode]
        dev = q.device
        if indices_out is None:
            indices_out = torch.empty((T, 1, topk), dtype=torch.int32, device=dev)
        if mode == 2 and cand_out is None:
            cand_out = torch.empty((T, 1, cand_blocks), dtype=torch.int32, device=dev)
        a = Args()
        a.q = _ptr(q); a.q_stride_t = q.stride(0); a.q_stride_h = q.stride(1)
        a.T, a.N, a.D = T, N, D
        a.cu_seqlens_q = _ptr(cu_seqlens_q); a.B = B
        a.k_lens = _ptr(k_lens); a.residual = _ptr(residual)
        a.cache = _ptr(cache); a.page_stride = page_stride; a.rows_per_page = rows_per_page
        a.k_offset = k_offset; a.scale_offset = scale_offset
        a.num_pages = cache.numel() // page_stride
        a.block_table = _ptr(block_table); a.bt_stride = block_table.stride(0)
        a.head_weights = _ptr(head_weights); a.q_scale = _ptr(q_scale)
        a.ratio = ratio; a.mask_mode = MASK_CAUSAL; a.quant_mode = quant_mode
        a.layout_q = LAYOUT_TND; a.layout_k = LAYOUT_PA_BBND
        a.topk = topk; a.cand_mode = mode; a.cand_blocks = cand_blocks; a.block_size = 8
        a.cand_in = _ptr(cand_in); a.cand_in_numel = 0 if cand_in is None else cand_in.numel()
        a.cand_out = _ptr(cand_out); a.cand_out_numel = 0 if cand_out is None else cand_out.numel()
        a.indices_out = _ptr(indices_out); a.indices_numel = indices_out.numel()
        self.args = a
        self.keep = (q, cu_seqlens_q, k_lens, residual, cache, block_table, head_weights,
                     q_scale, cand_in)
        self.indices = indices_out
        self.cand = cand_out
        self.device = dev

    def workspace_bytes(self) -> int:
        n = c_size_t(0)
        _check(lib().qli_workspace_size(ctypes.byref(self.args), ctypes.byref(n)),
               "qli_workspace_size")
        return int(n.value)

    def alloc_workspace(self):
        import torch
        n = max(256, self.workspace_bytes())
        return torch.empty(n, dtype=torch.uint8, device=self.device)

    def run(self, workspace, stream=None):
        _check(lib().qli_run(ctypes.byref(self.args), _ptr(workspace), workspace.numel(),
                             _stream(stream)), "qli_run")
        return self.indices, self.cand

    def run_static(self, stream=None):
        """qli_run_static: the same call on the library's fixed scratch array
        (for callers that cannot allocate a workspace)."""
        _check(lib().qli_run_static(ctypes.byref(self.args), _stream(stream)), "qli_run_static")
        return self.indices, self.cand

    def static_device_error(self, stream=None) -> int:
        """The device error word of the last run_static call on this device."""
        w = c_uint32(0)
        _check(lib().qli_read_static_device_error(ctypes.byref(w), _stream(stream)),
               "qli_read_static_device_error")
        return int(w.value)

    def run_stage(self, stage: int, workspace, stream=None):
        _check(lib().qli_run_stage(ctypes.byref(self.args), _ptr(workspace), workspace.numel(),
                                   stage, _stream(stream)), "qli_run_stage")

    def launches(self, stage: int = 0) -> int:
        n = c_int32(0)
        _check(lib().qli_launch_count(ctypes.byref(self.args), stage, ctypes.byref(n)),
               "qli_launch_count")
        return int(n.value)

    def scores(self, workspace):
        """FP32 score rows the SCORE stage left in the workspace: [T, row_stride]."""
        import torch
        off, stride = c_size_t(0), c_int64(0)
        _check(lib().qli_scores_layout(ctypes.byref(self.args), ctypes.byref(off),
                                       ctypes.byref(stride)), "qli_scores_layout")
        T = self.args.T
        n = T * stride.value
        view = workspace[off.value:off.value + 4 * n].view(torch.float32)
        return view.view(T, stride.value)

    def device_error(self, workspace, stream=None) -> int:
        w = c_uint32(0)
        _check(lib().qli_read_device_error(_ptr(workspace), ctypes.byref(w), _stream(stream)),
               "qli_read_device_error")
        return int(w.value)


def _stream(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def run(*args, workspace=None, stream=None, **kw):
    """One indexer call. Returns (indices [T,1,K] int32, candidates [T,1,C] int32 or None)."""
    c = Call(*args, **kw)
    ws = c.alloc_workspace() if workspace is None else workspace
    return c.run(ws, stream)


def quantize_q(x, q_out=None, scale_out=None, stream=None, quant_mode=QUANT_INT8):
    """qli_quantize_q (or, with quant_mode=QUANT_FP8, qli_quantize_q_fp8): BF16
    rows x [..., 128] (torch.bfloat16 or int16/uint16 bit patterns, CUDA,
    contiguous) -> (codes int8 [..., 128] (E4M3 bit patterns for FP8), FP16
    scale bits int16 [...]). For the indexer's queries x is [T, N, 128]."""
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA tensor")
    if x.element_size() != 2 or x.shape[-1] != 128:
        raise TypeError("x must hold 16-bit BF16 patterns with 128 values per row")
    rows = x.numel() // 128
    if q_out is None:
        q_out = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scale_out is None:
        scale_out = torch.empty(x.shape[:-1], dtype=torch.int16, device=x.device)
    _require_cuda("q_out", q_out, torch.int8)
    name = "qli_quantize_q_fp8" if quant_mode == QUANT_FP8 else "qli_quantize_q"
    _check(getattr(lib(), name)(_ptr(x), rows, _ptr(q_out), _ptr(scale_out), _stream(stream)),
           name)
    return q_out, scale_out


def check_quant_rounding(stream=None):
    """qli_check_quant_rounding: (code mismatches, quotient mismatches) of
    the quantisers' division against IEEE FP32 division over every BF16 x and
    every positive finite FP16 scale."""
    import torch
    counts = torch.empty(2, dtype=torch.int64, device="cuda")
    _check(lib().qli_check_quant_rounding(_ptr(counts), _stream(stream)),
           "qli_check_quant_rounding")
    return tuple(int(v) for v in counts.cpu())


def write_index_k(k, slot_mapping, cache, *, rows_per_page: int, page_stride: int,
                  k_offset: int, scale_offset: int, err_word=None, stream=None,
                  quant_mode=QUANT_INT8):
    """qli_write_index_k (or, with quant_mode=QUANT_FP8, qli_write_index_k_fp8):
    quantises the rows of k [n, 128] (BF16 patterns, CUDA, contiguous) and
    writes them into the page pool `cache` (uint8, CUDA) at slot_mapping [n]
    (int64: page * rows_per_page + row; negative = skip)."""
    import torch
    _require_cuda("slot_mapping", slot_mapping, torch.int64)
    _require_cuda("cache", cache, torch.uint8)
    _require_cuda("err_word", err_word, torch.int32)
    if not isinstance(k, torch.Tensor) or not k.is_cuda or not k.is_contiguous() \
            or k.element_size() != 2 or k.dim() != 2 or k.shape[1] != 128:
        raise TypeError("k must be a contiguous CUDA [n, 128] tensor of BF16 patterns")
    if slot_mapping.numel() != k.shape[0]:
        raise ValueError("one slot per row")
    num_pages = cache.numel() // page_stride
    name = "qli_write_index_k_fp8" if quant_mode == QUANT_FP8 else "qli_write_index_k"
    _check(getattr(lib(), name)(_ptr(k), k.shape[0], _ptr(slot_mapping), _ptr(cache), num_pages,
                                page_stride, rows_per_page, k_offset, scale_offset,
                                _ptr(err_word), _stream(stream)), name)


def sparse_attention(q, cu_seqlens_q, cache, block_table, indices, *, rows_per_page: int,
                     page_stride: int, scale: float, kv_offset: int = 0, out=None, lse=None,
                     err_word=None, stream=None):
    """qli_sparse_attention: softmax attention of q [T, H, 512] (BF16, CUDA)
    over the KV rows of the positions in indices [T, 1, K] (int32, -1
    skipped), read through block_table from the page pool `cache`. Returns
    (out [T, H, 512] BF16, lse [T, H] float32)."""
    import torch
    _require_cuda("q", q, torch.bfloat16)
    _require_cuda("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _require_cuda("cache", cache, torch.uint8)
    _require_cuda("block_table", block_table, torch.int32)
    _require_cuda("indices", indices, torch.int32)
    _require_cuda("err_word", err_word, torch.int32)
    if q.dim() != 3 or q.stride(2) != 1:
        raise ValueError("q must be [T, H, 512] with unit stride in the last dim")
    if not indices.is_contiguous() or indices.dim() != 3:
        raise ValueError("indices must be a contiguous [T, 1, K] tensor")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [B, bt_stride] row-major")
    T, H, D = q.shape
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _require_cuda("out", out, torch.bfloat16)
    _require_cuda("lse", lse, torch.float32)
    if out.stride(2) != 1 or not lse.is_contiguous():
        raise ValueError("out must have unit stride in the last dim and lse be contiguous")
    a = AttnArgs()
    a.q = _ptr(q); a.q_stride_t = q.stride(0); a.q_stride_h = q.stride(1)
    a.T, a.H, a.D = T, H, D
    a.cu_seqlens_q = _ptr(cu_seqlens_q); a.B = cu_seqlens_q.numel() - 1
    a.cache = _ptr(cache); a.page_stride = page_stride; a.num_pages = cache.numel() // page_stride
    a.rows_per_page = rows_per_page; a.kv_offset = kv_offset
    a.block_table = _ptr(block_table); a.bt_stride = block_table.stride(0)
    a.indices = _ptr(indices); a.K = indices.shape[-1]; a.scale = float(scale)
    a.out = _ptr(out); a.out_stride_t = out.stride(0); a.out_stride_h = out.stride(1)
    a.lse = _ptr(lse); a.err_word = _ptr(err_word)
    _check(lib().qli_sparse_attention(ctypes.byref(a), _stream(stream)), "qli_sparse_attention")
    return out, lse

