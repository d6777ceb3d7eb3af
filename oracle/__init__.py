"""fp64 CPU oracle for the DeepSeek sparse-attention decode path.

TEST INFRASTRUCTURE ONLY: this package is the checker, not the product.  Only
the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  The CUDA library never links, loads or calls it, and it shares no
code with the CUDA sources.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc and exposes numpy-facing wrappers.  Functions
and the passages they follow:

* ``decode_e4m3 / decode_e2m1 / decode_ue8m0 / decode_bf16`` -- the OCP FP8,
  FP4 and UE8M0 definitions and bfloat16 (upper half of binary32).
* ``visible`` -- draft-row windows ("feat(deepseek_v4): Add fp4 indexer for
  dsv4", varlen windows per draft row; reading: L - next_n + i + 1, clamped),
  over a compressed cache floor(window / ratio) entries (the CSA index length
  context_len // 4 of the same page).
* ``logits_fp8 / logits_mxfp4`` -- the lightning-indexer score
  k_scale[s] * sum_h w[r,h] * relu(q[r,h].k[s]) over a paged cache
  ("SM120 FP8 paged MQA page 32", Summary; "Add fp4 indexer for dsv4", FP4
  mqa-logits).
* ``topk`` -- full sort, descending logit, ties by ascending index, -1 padding.
* ``sparse_mla`` -- softmax attention over the selected latent tokens with an
  fp32-style LSE output ("Add DeepSeek V4 sparse MLA TRTLLM-GEN kernels").
* ``sparse_mla_swa`` -- sparse MLA over the selected entries of one latent
  cache plus a sliding window of another in one softmax, with per-row top-k
  lengths and cumulative query lengths ("Add DeepSeek V4 sparse MLA TRTLLM-GEN
  kernels": sliding_window_kv_cache, sparse_topk_lens, cum_seq_lens_q).
* ``encode_e4m3 / encode_e2m1 / quantize_scatter`` -- writing new K rows into
  the paged FP8 (per-token fp32 scale) or MXFP4 (ue8m0 per 32 elements) cache
  through a slot mapping ("feat(deepseek_v4): Add fp4 indexer for dsv4": the FP4
  indexer's cache scatter beside its logits kernel; OCP MX v1.0 block scaling).

Parity pins: tests/test_oracle_*.py.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_FP8 = 0
FMT_BF16 = 2

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_u8p = ctypes.POINTER(ctypes.c_uint8)
_c_f32p = ctypes.POINTER(ctypes.c_float)
_c_f64p = ctypes.POINTER(ctypes.c_double)
_c_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.dsa_oracle_e4m3.restype = ctypes.c_double
        lib.dsa_oracle_e4m3.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_e2m1.restype = ctypes.c_double
        lib.dsa_oracle_e2m1.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_ue8m0.restype = ctypes.c_double
        lib.dsa_oracle_ue8m0.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_bf16.restype = ctypes.c_double
        lib.dsa_oracle_bf16.argtypes = [ctypes.c_uint16]
        lib.dsa_oracle_visible.restype = _int
        lib.dsa_oracle_visible.argtypes = [_int, _int, _int]
        lib.dsa_oracle_logits_fp8.restype = _int
        lib.dsa_oracle_logits_fp8.argtypes = [
            _c_u8p, _c_f32p, _int, _int, _c_u8p, _i64, _i64, _c_u8p, _i64, _i64,
            _c_i32p, _i64, _int, _int, _int, _c_i32p, _int, _int, _int, _int, _int,
            _c_f64p, _i64, _int]
        lib.dsa_oracle_logits_mxfp4.restype = _int
        lib.dsa_oracle_logits_mxfp4.argtypes = [
            _c_u8p, _c_u8p, _c_f32p, _int, _int, _c_u8p, _i64, _i64, _c_u8p, _i64, _i64,
            _c_i32p, _i64, _int, _int, _int, _c_i32p, _int, _int, _int, _int, _int,
            _c_f64p, _i64, _int]
        lib.dsa_oracle_topk.restype = _int
        lib.dsa_oracle_topk.argtypes = [
            _c_f64p, _i64, _c_i32p, _int, _int, _int, _int, _int, _int, _c_i32p, _i64, _c_i32p]
        lib.dsa_oracle_sparse_mla.restype = _int
        lib.dsa_oracle_sparse_mla.argtypes = [
            _c_u16p, _int, _int, _int, _int, ctypes.c_double, _int, _c_u8p, _i64, _i64,
            _c_u8p, _i64, _i64, _c_i32p, _i64, _int, _int, _int, _c_i32p, _int,
            _c_i32p, _i64, _int, _c_f64p, _c_f64p]
        lib.dsa_oracle_sparse_mla_swa.restype = _int
        lib.dsa_oracle_sparse_mla_swa.argtypes = [
            _c_u16p, _int, _int, _int, _int, ctypes.c_double, _int,
            _c_u8p, _i64, _i64, _c_u8p, _i64, _i64, _c_i32p, _i64, _int, _int, _int,
            _c_i32p, _i64, _int, _c_i32p,
            _c_u8p, _i64, _i64, _c_u8p, _i64, _i64, _c_i32p, _i64, _int, _int, _int, _int,
            _c_i32p, _c_i32p, _int, _int, _c_f64p, _c_f64p]
        lib.dsa_oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.dsa_oracle_encode_e4m3.argtypes = [ctypes.c_float]
        lib.dsa_oracle_encode_e2m1.restype = ctypes.c_uint8
        lib.dsa_oracle_encode_e2m1.argtypes = [ctypes.c_float]
        lib.dsa_oracle_quantize_scatter.restype = _int
        lib.dsa_oracle_quantize_scatter.argtypes = [
            ctypes.c_void_p, _int, _i64, _int, _int, ctypes.POINTER(ctypes.c_int64), _int,
            _c_u8p, _i64, _i64, _c_u8p, _i64, _i64, _int, _int]
        lib.dsa_oracle_threads.restype = _int
        lib.dsa_oracle_threads.argtypes = []
        _lib = lib
        return lib


def _np(x, dtype):
    """numpy view of a CPU torch tensor or numpy array, C-contiguous, given dtype."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != dtype:
        x = x.view(dtype) if x.dtype.itemsize == np.dtype(dtype).itemsize else x.astype(dtype)
    return x


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def threads() -> int:
    return _load().dsa_oracle_threads()


def decode_e4m3(code: int) -> float:
    return _load().dsa_oracle_e4m3(code)


def decode_e2m1(nibble: int) -> float:
    return _load().dsa_oracle_e2m1(nibble)


def decode_ue8m0(code: int) -> float:
    return _load().dsa_oracle_ue8m0(code)


def decode_bf16(bits: int) -> float:
    return _load().dsa_oracle_bf16(bits)


def visible(L: int, next_n: int, i: int, ratio: int = 1) -> int:
    """Entries row i sees: floor(clamp(L - next_n + i + 1, 0, L) / ratio)."""
    return _load().dsa_oracle_visible(L, next_n, i) // int(ratio)


class PagedBytes:
    """A paged cache seen as raw bytes: ``values``/``scales`` are flat uint8
    buffers; token ``t`` of physical page ``p`` starts at ``p*page_stride +
    t*token_stride`` bytes in each.  ``block_table`` is [batch, max_pages] int32."""

    def __init__(self, values, val_page_stride, val_token_stride, scales, sc_page_stride,
                 sc_token_stride, block_table, page_kv, num_pages):
        self.values = _np(values, np.uint8).reshape(-1)
        self.vps = int(val_page_stride)
        self.vts = int(val_token_stride)
        self.scales = None if scales is None else _np(scales, np.uint8).reshape(-1)
        self.sps = int(sc_page_stride)
        self.sts = int(sc_token_stride)
        bt = _np(block_table, np.int32)
        self.block_table = bt.reshape(bt.shape[0], -1)
        self.page_kv = int(page_kv)
        self.num_pages = int(num_pages)


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s failed with code %d" % (what, rc))


def logits_fp8(q, w, cache: PagedBytes, context_lens, next_n, row_begin=None, row_end=None,
               width=None, ratio=1):
    """fp64 logits [row_end-row_begin, width]; entries past each row's visible
    length are NaN (not defined by the method)."""
    lib = _load()
    q = _np(q, np.uint8)
    R, H, D = q.shape
    w = _np(w, np.float32).reshape(R, H)
    ctx = _np(context_lens, np.int32).reshape(-1)
    batch = ctx.shape[0]
    rb = 0 if row_begin is None else int(row_begin)
    re = batch * next_n if row_end is None else int(row_end)
    if width is None:
        width = int(max([0] + [lib.dsa_oracle_visible(int(L), next_n, next_n - 1) // int(ratio) for L in ctx]))
    out = np.full((max(re - rb, 0), max(width, 1)), np.nan, dtype=np.float64)
    bt = cache.block_table
    rc = lib.dsa_oracle_logits_fp8(
        _ptr(q, ctypes.c_uint8), _ptr(w, ctypes.c_float), H, D,
        _ptr(cache.values, ctypes.c_uint8), cache.vps, cache.vts,
        _ptr(cache.scales, ctypes.c_uint8), cache.sps, cache.sts,
        _ptr(bt, ctypes.c_int32), bt.shape[1], bt.shape[1], cache.page_kv, cache.num_pages,
        _ptr(ctx, ctypes.c_int32), batch, int(next_n), int(ratio), rb, re,
        _ptr(out, ctypes.c_double), out.shape[1], int(width))
    _check(rc, "logits_fp8")
    return out[:, :width]


def logits_mxfp4(q, q_scales, w, cache: PagedBytes, context_lens, next_n, row_begin=None,
                 row_end=None, width=None, ratio=1):
    """fp64 logits for an MXFP4 cache and MXFP4 q (packed e2m1 + ue8m0 per 32)."""
    lib = _load()
    q = _np(q, np.uint8)
    R, H, Dh = q.shape
    D = 2 * Dh
    qs = _np(q_scales, np.uint8).reshape(R, H, D // 32)
    w = _np(w, np.float32).reshape(R, H)
    ctx = _np(context_lens, np.int32).reshape(-1)
    batch = ctx.shape[0]
    rb = 0 if row_begin is None else int(row_begin)
    re = batch * next_n if row_end is None else int(row_end)
    if width is None:
        width = int(max([0] + [lib.dsa_oracle_visible(int(L), next_n, next_n - 1) // int(ratio) for L in ctx]))
    out = np.full((max(re - rb, 0), max(width, 1)), np.nan, dtype=np.float64)
    bt = cache.block_table
    rc = lib.dsa_oracle_logits_mxfp4(
        _ptr(q, ctypes.c_uint8), _ptr(qs, ctypes.c_uint8), _ptr(w, ctypes.c_float), H, D,
        _ptr(cache.values, ctypes.c_uint8), cache.vps, cache.vts,
        _ptr(cache.scales, ctypes.c_uint8), cache.sps, cache.sts,
        _ptr(bt, ctypes.c_int32), bt.shape[1], bt.shape[1], cache.page_kv, cache.num_pages,
        _ptr(ctx, ctypes.c_int32), batch, int(next_n), int(ratio), rb, re,
        _ptr(out, ctypes.c_double), out.shape[1], int(width))
    _check(rc, "logits_mxfp4")
    return out[:, :width]


def topk(logits, context_lens, next_n, k, row_begin=None, row_end=None, ratio=1):
    """(idx [rows, k] int32 in sorted order with -1 padding, count [rows] int32)."""
    lib = _load()
    lg = np.ascontiguousarray(_np(logits, np.float64))
    ctx = _np(context_lens, np.int32).reshape(-1)
    batch = ctx.shape[0]
    rb = 0 if row_begin is None else int(row_begin)
    re = batch * next_n if row_end is None else int(row_end)
    rows = re - rb
    if lg.ndim == 1:
        lg = lg.reshape(rows, -1)
    idx = np.empty((rows, k), dtype=np.int32)
    cnt = np.empty((rows,), dtype=np.int32)
    rc = lib.dsa_oracle_topk(_ptr(lg, ctypes.c_double), lg.shape[1], _ptr(ctx, ctypes.c_int32),
                             batch, int(next_n), int(ratio), rb, re, int(k), _ptr(idx, ctypes.c_int32), k,
                             _ptr(cnt, ctypes.c_int32))
    _check(rc, "topk")
    return idx, cnt


def sparse_mla(q_bf16, softmax_scale, fmt, cache: PagedBytes, idx, d_v, seq_of_row=None,
               next_n=1):
    """(out [rows, Hq, d_v] fp64, lse [rows, Hq] fp64).  q_bf16 holds bf16 bits
    ([rows, Hq, d_qk] uint16 / int16 / torch.bfloat16)."""
    lib = _load()
    if hasattr(q_bf16, "dtype") and str(q_bf16.dtype) == "torch.bfloat16":
        q_bf16 = q_bf16.view(__import__("torch").int16)
    q = _np(q_bf16, np.uint16)
    rows, Hq, d_qk = q.shape
    ix = _np(idx, np.int32).reshape(rows, -1)
    k = ix.shape[1]
    out = np.zeros((rows, Hq, d_v), dtype=np.float64)
    lse = np.zeros((rows, Hq), dtype=np.float64)
    bt = cache.block_table
    sor = None if seq_of_row is None else _np(seq_of_row, np.int32).reshape(-1)
    sc = cache.scales if cache.scales is not None else np.zeros(16, np.uint8)
    rc = lib.dsa_oracle_sparse_mla(
        _ptr(q, ctypes.c_uint16), rows, Hq, d_qk, int(d_v), float(softmax_scale), int(fmt),
        _ptr(cache.values, ctypes.c_uint8), cache.vps, cache.vts,
        _ptr(sc, ctypes.c_uint8), cache.sps, cache.sts,
        _ptr(bt, ctypes.c_int32), bt.shape[1], bt.shape[1], cache.page_kv, cache.num_pages,
        None if sor is None else _ptr(sor, ctypes.c_int32), int(next_n),
        _ptr(ix, ctypes.c_int32), k, k, _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    _check(rc, "sparse_mla")
    return out, lse


def encode_e4m3(v: float) -> int:
    """Nearest e4m3 code to the float32 value v (ties to even, saturating)."""
    return int(_load().dsa_oracle_encode_e4m3(float(v)))


def encode_e2m1(v: float) -> int:
    """Nearest e2m1 code (4 bits) to the float32 value v (ties to even, saturating)."""
    return int(_load().dsa_oracle_encode_e2m1(float(v)))


def quantize_scatter(k, slots, fmt, cache: PagedBytes):
    """Quantise rows of new K (fp32 array, or torch bf16 / fp32 tensor) and write
    them into ``cache`` (its values / scales byte buffers are updated in place)
    at the physical slots ``slots`` (int64, page * page_kv + row; < 0 skipped).
    fmt: 0 = FP8 e4m3 + fp32 token scale, 1 = MXFP4 (e2m1 + ue8m0 per 32)."""
    lib = _load()
    is_bf16 = hasattr(k, "dtype") and str(k.dtype) == "torch.bfloat16"
    if is_bf16:
        arr = _np(k.view(__import__("torch").int16), np.uint16)
    else:
        arr = _np(k, np.float32)
    n, D = arr.shape
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64).reshape(-1))
    assert sl.shape[0] == n
    rc = lib.dsa_oracle_quantize_scatter(
        arr.ctypes.data_as(ctypes.c_void_p), 1 if is_bf16 else 0, D, n, D,
        sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(fmt),
        _ptr(cache.values, ctypes.c_uint8), cache.vps, cache.vts,
        _ptr(cache.scales, ctypes.c_uint8), cache.sps, cache.sts, cache.page_kv, cache.num_pages)
    _check(rc, "quantize_scatter")


def sparse_mla_swa(q_bf16, softmax_scale, fmt, cache: PagedBytes, idx, d_v, seq_lens, topk_lens=None,
                   swa: PagedBytes = None, window=0, cum_q=None, next_n=1):
    """(out [rows, Hq, d_v] fp64, lse [rows, Hq] fp64) of sparse MLA over the
    first topk_lens[r] entries of idx (cache ``cache``) plus the last
    min(window, vis) visible positions of the window cache ``swa``, in one
    softmax.  Rows map to sequences through cum_q ([batch + 1]) or r / next_n."""
    lib = _load()
    if hasattr(q_bf16, "dtype") and str(q_bf16.dtype) == "torch.bfloat16":
        q_bf16 = q_bf16.view(__import__("torch").int16)
    q = _np(q_bf16, np.uint16)
    rows, Hq, d_qk = q.shape
    ix = _np(idx, np.int32).reshape(rows, -1)
    k = ix.shape[1]
    sl = _np(seq_lens, np.int32).reshape(-1)
    batch = sl.shape[0]
    tl = None if topk_lens is None else _np(topk_lens, np.int32).reshape(-1)
    cq = None if cum_q is None else _np(cum_q, np.int32).reshape(-1)
    out = np.zeros((rows, Hq, d_v), dtype=np.float64)
    lse = np.zeros((rows, Hq), dtype=np.float64)
    bt = cache.block_table
    sc = cache.scales if cache.scales is not None else np.zeros(16, np.uint8)
    if swa is not None:
        wbt = swa.block_table
        wsc = swa.scales if swa.scales is not None else np.zeros(16, np.uint8)
        wargs = (_ptr(swa.values, ctypes.c_uint8), swa.vps, swa.vts, _ptr(wsc, ctypes.c_uint8), swa.sps, swa.sts,
                 _ptr(wbt, ctypes.c_int32), wbt.shape[1], wbt.shape[1], swa.page_kv, swa.num_pages, int(window))
    else:
        wargs = (None, 0, 0, None, 0, 0, None, 0, 0, 0, 0, 0)
    rc = lib.dsa_oracle_sparse_mla_swa(
        _ptr(q, ctypes.c_uint16), rows, Hq, d_qk, int(d_v), float(softmax_scale), int(fmt),
        _ptr(cache.values, ctypes.c_uint8), cache.vps, cache.vts, _ptr(sc, ctypes.c_uint8), cache.sps, cache.sts,
        _ptr(bt, ctypes.c_int32), bt.shape[1], bt.shape[1], cache.page_kv, cache.num_pages,
        _ptr(ix, ctypes.c_int32), k, k, None if tl is None else _ptr(tl, ctypes.c_int32),
        *wargs, _ptr(sl, ctypes.c_int32), None if cq is None else _ptr(cq, ctypes.c_int32), batch, int(next_n),
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    _check(rc, "sparse_mla_swa")
    return out, lse
