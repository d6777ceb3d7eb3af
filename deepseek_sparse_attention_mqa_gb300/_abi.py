"""ctypes binding of libdsa (include/dsa.h): argument marshalling only.

Every function here passes device pointers, sizes and the current CUDA stream
to the C ABI and raises ``DSAError`` on a non-zero status.  No computation of
the path happens in Python; if libdsa.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CAPACITY, DSA_ERR_CUDA = range(5)
FMT_FP8, FMT_MXFP4, FMT_BF16 = 0, 1, 2
DEV_BAD_PAGE, DEV_WIDTH, DEV_TIMEOUT, DEV_BAD_INDEX, DEV_SCHEDULE = 0x1, 0x2, 0x4, 0x8, 0x10

# every symbol include/dsa.h declares
EXPORTS = (
    "dsa_status_string", "dsa_last_cuda_error", "dsa_version", "dsa_indexer_schedule_bytes",
    "dsa_indexer_build_schedule", "indexer_mqa_logits_paged", "dsa_topk_workspace_bytes",
    "indexer_topk", "dsa_sparse_mla_workspace_bytes", "sparse_mla_decode", "dsa_get_device_status",
    "indexer_mqa_logits_paged_noalloc", "dsa_wait_selftest", "dsa_kv_quantize_scatter",
    "dsa_score_topk_workspace_bytes", "indexer_score_topk", "sparse_mla_decode_swa",
)
DTYPE_F32, DTYPE_BF16 = 0, 1


class DSAError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = _lib.dsa_status_string(status).decode() if _lib is not None else str(status)
        msg = "%s failed: %s" % (what, name)
        if cuda_error:
            msg += " (cudaError %d)" % cuda_error
        super().__init__(msg)


class PagedCache(ctypes.Structure):
    """dsa_paged_cache."""
    _fields_ = [
        ("fmt", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_kv", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("values", ctypes.c_void_p),
        ("val_page_stride", ctypes.c_int64), ("val_token_stride", ctypes.c_int64),
        ("scales", ctypes.c_void_p), ("sc_page_stride", ctypes.c_int64),
        ("sc_token_stride", ctypes.c_int64), ("block_table", ctypes.c_void_p),
        ("bt_row_stride", ctypes.c_int64), ("max_pages_per_seq", ctypes.c_int32),
        ("compress_ratio", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


def lib():
    """Load libdsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdsa.so is not built (%s); run "
                               "deepseek_sparse_attention_mqa_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        L.dsa_status_string.restype = ctypes.c_char_p
        L.dsa_status_string.argtypes = [_i]
        L.dsa_last_cuda_error.restype = _i
        L.dsa_last_cuda_error.argtypes = []
        L.dsa_version.restype = _i
        L.dsa_version.argtypes = []
        L.dsa_indexer_schedule_bytes.restype = _sz
        L.dsa_indexer_schedule_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.dsa_indexer_build_schedule.restype = _i
        L.dsa_indexer_build_schedule.argtypes = [_vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp]
        L.indexer_mqa_logits_paged.restype = _i
        L.indexer_mqa_logits_paged.argtypes = [
            _vp, _vp, _i, _vp, _i, ctypes.POINTER(PagedCache), _vp, _i, _i, _i, _i, _vp, _sz,
            _vp, _i64, _i, _vp, _vp]
        L.indexer_mqa_logits_paged_noalloc.restype = _i
        L.indexer_mqa_logits_paged_noalloc.argtypes = [
            _vp, _vp, _i, _vp, _i, ctypes.POINTER(PagedCache), _vp, _i, _i, _i, _i, _vp, _i64, _i,
            _vp, _vp]
        L.dsa_topk_workspace_bytes.restype = _sz
        L.dsa_topk_workspace_bytes.argtypes = [_i, _i, _i]
        L.indexer_topk.restype = _i
        L.indexer_topk.argtypes = [_vp, _i64, _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _i64, _vp, _vp,
                                   _sz, _vp, _vp]
        L.dsa_sparse_mla_workspace_bytes.restype = _sz
        L.dsa_sparse_mla_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.sparse_mla_decode.restype = _i
        L.sparse_mla_decode.argtypes = [_vp, _i, _i, _i, _i, ctypes.c_float,
                                        ctypes.POINTER(PagedCache), _vp, _i, _vp, _i64, _i, _vp,
                                        _vp, _vp, _sz, _vp, _vp]
        L.dsa_score_topk_workspace_bytes.restype = _sz
        L.dsa_score_topk_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.indexer_score_topk.restype = _i
        L.indexer_score_topk.argtypes = [
            _vp, _vp, _i, _vp, _i, ctypes.POINTER(PagedCache), _vp, _i, _i, _i, _i, _vp, _sz,
            _vp, _i64, _i, _i, _vp, _i64, _vp, _vp, _sz, _vp, _vp]
        L.dsa_kv_quantize_scatter.restype = _i
        L.dsa_kv_quantize_scatter.argtypes = [_vp, _i, _i64, _i, _vp, ctypes.POINTER(PagedCache), _vp, _vp]
        L.dsa_wait_selftest.restype = _i
        L.dsa_wait_selftest.argtypes = [_vp, ctypes.c_int32, _i, _vp, _vp]
        L.sparse_mla_decode_swa.restype = _i
        L.sparse_mla_decode_swa.argtypes = [
            _vp, _i, _i, _i, _i, ctypes.c_float, ctypes.POINTER(PagedCache), _vp, _i64, _i, _vp,
            ctypes.POINTER(PagedCache), _i, _vp, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp, _vp]
        L.dsa_get_device_status.restype = _i
        L.dsa_get_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32), _vp]
        _lib = L
        return L


def _check(st: int, what: str):
    if st != DSA_OK:
        raise DSAError(st, what, lib().dsa_last_cuda_error() if st == DSA_ERR_CUDA else 0)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_cache(fmt, head_dim, page_kv, num_pages, values, val_page_stride, val_token_stride,
               scales, sc_page_stride, sc_token_stride, block_table, compress_ratio=1) -> PagedCache:
    """dsa_paged_cache over device tensors (block_table [batch, max_pages] int32);
    compress_ratio = tokens per entry of a compressed indexer cache."""
    c = PagedCache()
    c.fmt, c.head_dim, c.page_kv, c.num_pages = int(fmt), int(head_dim), int(page_kv), int(num_pages)
    c.values = values.data_ptr()
    c.val_page_stride, c.val_token_stride = int(val_page_stride), int(val_token_stride)
    c.scales = None if scales is None else scales.data_ptr()
    c.sc_page_stride, c.sc_token_stride = int(sc_page_stride), int(sc_token_stride)
    c.block_table = block_table.data_ptr()
    c.bt_row_stride = int(block_table.stride(0))
    c.max_pages_per_seq = int(block_table.shape[1])
    c.compress_ratio = int(compress_ratio)
    c._keep = (values, scales, block_table)
    return c


def schedule_bytes(batch, next_n, num_heads, row_begin, row_end) -> int:
    return int(lib().dsa_indexer_schedule_bytes(batch, next_n, num_heads, row_begin, row_end))


def build_schedule(context_lens, batch, next_n, num_heads, row_begin, row_end, sched,
                   status=None, stream=None, compress_ratio=1):
    _check(lib().dsa_indexer_build_schedule(
        _ptr(context_lens), batch, next_n, num_heads, int(compress_ratio), row_begin, row_end, _ptr(sched),
        sched.numel() * sched.element_size(), _ptr(status), _stream(stream)),
        "dsa_indexer_build_schedule")


def mqa_logits(q, q_scales, fmt, weights, num_heads, cache: PagedCache, context_lens, batch,
               next_n, row_begin, row_end, sched, logits, logits_width, status=None, stream=None):
    """indexer_mqa_logits_paged; ``sched=None`` lets the kernel build the units of
    a call with at most INLINE_UNITS units itself (no schedule launch)."""
    _check(lib().indexer_mqa_logits_paged(
        _ptr(q), _ptr(q_scales), int(fmt), _ptr(weights), num_heads, ctypes.byref(cache),
        _ptr(context_lens), batch, next_n, row_begin, row_end, _ptr(sched),
        0 if sched is None else sched.numel() * sched.element_size(), _ptr(logits), logits.stride(0),
        int(logits_width), _ptr(status), _stream(stream)), "indexer_mqa_logits_paged")


INLINE_UNITS = 256      # kInlineUnits of the library


def score_topk_workspace_bytes(batch, next_n, num_heads, row_begin, row_end) -> int:
    return int(lib().dsa_score_topk_workspace_bytes(batch, next_n, num_heads, row_begin, row_end))


def score_topk(q, q_scales, fmt, weights, num_heads, cache: PagedCache, context_lens, batch, next_n,
               row_begin, row_end, sched, logits, logits_width, k, idx, count, workspace, status=None,
               stream=None):
    """indexer_score_topk: logits and the per-row top-k in one launch.
    ``workspace`` must be zero before the first call (the call leaves it zero)."""
    _check(lib().indexer_score_topk(
        _ptr(q), _ptr(q_scales), int(fmt), _ptr(weights), num_heads, ctypes.byref(cache),
        _ptr(context_lens), batch, next_n, row_begin, row_end, _ptr(sched),
        0 if sched is None else sched.numel() * sched.element_size(), _ptr(logits), logits.stride(0),
        int(logits_width), int(k), _ptr(idx), idx.stride(0), _ptr(count), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)), "indexer_score_topk")


def units_of(batch, next_n, num_heads, row_begin, row_end) -> int:
    """Work units of a logits call (rows of one sequence sharing an MMA)."""
    if row_end <= row_begin:
        return 0
    g = max(1, min(next_n, 256 // num_heads))
    total = 0
    b0, b1 = row_begin // next_n, (row_end - 1) // next_n
    for b in range(b0, min(b1, batch - 1) + 1):
        lo, hi = max(b * next_n, row_begin), min((b + 1) * next_n, row_end)
        total += (hi - lo + g - 1) // g
    return total


def mqa_logits_noalloc(q, q_scales, fmt, weights, num_heads, cache: PagedCache, context_lens,
                       batch, next_n, row_begin, row_end, logits, logits_width, status=None,
                       stream=None):
    """indexer_mqa_logits_paged_noalloc: the schedule lives in the library's fixed
    device array, so no schedule buffer is passed."""
    _check(lib().indexer_mqa_logits_paged_noalloc(
        _ptr(q), _ptr(q_scales), int(fmt), _ptr(weights), num_heads, ctypes.byref(cache),
        _ptr(context_lens), batch, next_n, row_begin, row_end, _ptr(logits), logits.stride(0),
        int(logits_width), _ptr(status), _stream(stream)), "indexer_mqa_logits_paged_noalloc")


def topk_workspace_bytes(rows, width, k) -> int:
    return int(lib().dsa_topk_workspace_bytes(rows, width, k))


def topk(logits, logits_width, context_lens, batch, next_n, row_begin, row_end, k, idx,
         count=None, workspace=None, status=None, stream=None, compress_ratio=1):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().indexer_topk(
        _ptr(logits), logits.stride(0), int(logits_width), _ptr(context_lens), batch, next_n,
        int(compress_ratio), row_begin, row_end, k, _ptr(idx), idx.stride(0), _ptr(count), _ptr(workspace), ws_bytes,
        _ptr(status), _stream(stream)), "indexer_topk")


def mla_workspace_bytes(rows, num_heads, d_qk, d_v, k) -> int:
    return int(lib().dsa_sparse_mla_workspace_bytes(rows, num_heads, d_qk, d_v, k))


def sparse_mla(q_bf16, softmax_scale, cache: PagedCache, idx, k, out, lse, d_v,
               seq_of_row=None, next_n=1, workspace=None, status=None, stream=None):
    rows, heads, d_qk = q_bf16.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sparse_mla_decode(
        _ptr(q_bf16), rows, heads, d_qk, int(d_v), float(softmax_scale), ctypes.byref(cache),
        _ptr(seq_of_row), next_n, _ptr(idx), idx.stride(0), int(k), _ptr(out), _ptr(lse),
        _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)), "sparse_mla_decode")


def device_status(status, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib().dsa_get_device_status(_ptr(status), ctypes.byref(v), _stream(stream)),
           "dsa_get_device_status")
    return int(v.value)


def wait_selftest(flag, expect, limit_us, status, stream=None):
    """dsa_wait_selftest: a bounded wait on a barrier arrived on only if
    flag[0] == expect; a wait that runs out sets DEV_TIMEOUT in status."""
    _check(lib().dsa_wait_selftest(_ptr(flag), int(expect), int(limit_us), _ptr(status),
                                   _stream(stream)), "dsa_wait_selftest")


def kv_quantize_scatter(k_new, slot_mapping, cache: PagedCache, status=None, stream=None):
    """dsa_kv_quantize_scatter: quantise rows of k_new ([n, D] float32 or
    bfloat16 device tensor) into `cache` at slot_mapping ([n] int64)."""
    import torch
    dt = DTYPE_BF16 if k_new.dtype == torch.bfloat16 else DTYPE_F32
    if k_new.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("k_new must be float32 or bfloat16")
    _check(lib().dsa_kv_quantize_scatter(
        _ptr(k_new), dt, k_new.stride(0) if k_new.dim() == 2 else k_new.shape[-1], k_new.shape[0],
        _ptr(slot_mapping), ctypes.byref(cache), _ptr(status), _stream(stream)), "dsa_kv_quantize_scatter")


def sparse_mla_swa(q_bf16, softmax_scale, cache: PagedCache, idx, k, out, lse, d_v, topk_lens=None,
                   swa: PagedCache = None, window=0, seq_lens=None, cum_q=None, batch=0, next_n=1,
                   status=None, stream=None):
    """sparse_mla_decode_swa: selected entries of `cache` plus the sliding window
    of `swa` in one softmax, per-row top-k lengths, varlen rows via cum_q."""
    rows, heads, d_qk = q_bf16.shape
    _check(lib().sparse_mla_decode_swa(
        _ptr(q_bf16), rows, heads, d_qk, int(d_v), float(softmax_scale), ctypes.byref(cache), _ptr(idx),
        idx.stride(0) if idx is not None else 0, int(k), _ptr(topk_lens),
        None if swa is None else ctypes.byref(swa), int(window), _ptr(seq_lens), _ptr(cum_q), int(batch),
        int(next_n), _ptr(out), _ptr(lse), None, 0, _ptr(status), _stream(stream)), "sparse_mla_decode_swa")
