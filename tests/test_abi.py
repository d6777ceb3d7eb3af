"""CPU checks of the C ABI: the library loads, exports every symbol that
include/dsa.h declares, and rejects bad arguments on the host before touching a
GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from deepseek_sparse_attention_mqa_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return _abi.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "dsa.h")).read()
    names = re.findall(r"^DSA_API\s+[\w\s\*]*?\b(\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) == len(_abi.EXPORTS)
    assert set(names) == set(_abi.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.dsa_status_string(0) == b"DSA_OK"
    assert L.dsa_status_string(3) == b"DSA_ERR_CAPACITY"
    assert L.dsa_version() >= 100


def test_paged_cache_struct_layout():
    # int32 x4, ptr, i64, i64, ptr, i64, i64, ptr, i64, int32, int32 = 88 bytes on LP64
    assert ctypes.sizeof(_abi.PagedCache) == 88
    assert _abi.PagedCache.values.offset == 16
    assert _abi.PagedCache.block_table.offset == 64
    assert _abi.PagedCache.max_pages_per_seq.offset == 80
    assert _abi.PagedCache.compress_ratio.offset == 84


def test_schedule_bytes_counts_units(L):
    # decode: one unit per sequence (64 heads -> at most 4 rows per unit, next_n 1)
    assert L.dsa_indexer_schedule_bytes(64, 1, 64, 0, 64) == 32 + 32 * 64
    # next_n 3 with 64 heads: 3 rows fit one MMA (192 columns) -> one unit per sequence
    assert L.dsa_indexer_schedule_bytes(5, 3, 64, 0, 15) == 32 + 32 * 5
    # prefill chunk: 4 rows per unit
    assert L.dsa_indexer_schedule_bytes(1, 16384, 64, 0, 8192) == 32 + 32 * 2048
    assert L.dsa_indexer_schedule_bytes(1, 16384, 64, 8192, 16384) == 32 + 32 * 2048
    # a range cutting through sequences: rows 2..9 of next_n 4 (H=128 -> 2 rows/unit)
    # seq0 rows 2,3 -> 1 unit; seq1 rows 4..7 -> 2 units; seq2 rows 8,9 -> 1 unit
    assert L.dsa_indexer_schedule_bytes(3, 4, 128, 2, 10) == 32 + 32 * 4
    # invalid row ranges give 0
    assert L.dsa_indexer_schedule_bytes(2, 1, 64, 0, 3) == 0
    assert L.dsa_indexer_schedule_bytes(2, 0, 64, 0, 0) == 0


def test_host_validation_rejects_before_any_gpu_call(L):
    vp = ctypes.c_void_p
    fake = vp(0x1000)   # never dereferenced: validation fails first
    # null schedule buffer
    assert L.dsa_indexer_build_schedule(fake, 2, 1, 64, 1, 0, 2, None, 4096, None, None) == 1
    # capacity
    assert L.dsa_indexer_build_schedule(fake, 2, 1, 64, 1, 0, 2, fake, 8, None, None) == 3
    # compression ratio out of range
    assert L.dsa_indexer_build_schedule(fake, 2, 1, 64, -2, 0, 2, fake, 4096, None, None) == 1
    # unsupported head count
    c = _abi.PagedCache()
    c.fmt, c.head_dim, c.page_kv, c.num_pages = 0, 128, 64, 4
    c.values, c.scales, c.block_table = 0x1000, 0x2000, 0x3000
    c.val_page_stride, c.val_token_stride = 64 * 128, 128
    c.sc_page_stride, c.sc_token_stride = 256, 4
    c.bt_row_stride, c.max_pages_per_seq = 4, 4
    args = lambda H, cache, width=256: (fake, None, 0, fake, H, ctypes.byref(cache), fake, 2, 1, 0,
                                        2, fake, 4096, fake, 256, width, None, None)
    assert L.indexer_mqa_logits_paged(*args(48, c)) == 2
    # page size outside {32, 64}
    c.page_kv = 128
    assert L.indexer_mqa_logits_paged(*args(64, c)) == 2
    c.page_kv = 64
    # misaligned page stride
    c.val_page_stride = 64 * 128 + 8
    assert L.indexer_mqa_logits_paged(*args(64, c)) == 1
    c.val_page_stride = 64 * 128
    # logits row stride smaller than the width
    assert L.indexer_mqa_logits_paged(*args(64, c, width=512)) == 1
    # format mismatch between q and cache
    a = list(args(64, c))
    a[2] = 1
    assert L.indexer_mqa_logits_paged(*a) == 2
    # top-k: k out of range, stride too small
    assert L.indexer_topk(fake, 256, 256, fake, 2, 1, 1, 0, 2, 0, fake, 64, None, None, 0, None, None) == 2
    assert L.indexer_topk(fake, 256, 256, fake, 2, 1, 1, 0, 2, 128, fake, 64, None, None, 0, None, None) == 1
    # MLA: d_v > d_qk, bad format
    m = _abi.PagedCache()
    m.fmt, m.head_dim, m.page_kv, m.num_pages = 0, 576, 64, 4
    m.values, m.scales, m.block_table = 0x1000, 0x2000, 0x3000
    m.val_page_stride, m.val_token_stride = 64 * 576, 576
    m.sc_page_stride, m.sc_token_stride = 256, 4
    m.bt_row_stride, m.max_pages_per_seq = 4, 4
    assert L.sparse_mla_decode(fake, 2, 128, 576, 640, 0.1, ctypes.byref(m), None, 1, fake, 64, 64,
                               fake, fake, None, 0, None, None) == 2
    m.fmt = 1
    assert L.sparse_mla_decode(fake, 2, 128, 576, 512, 0.1, ctypes.byref(m), None, 1, fake, 64, 64,
                               fake, fake, None, 0, None, None) == 2
    # device status read needs pointers
    assert L.dsa_get_device_status(None, None, None) == 1


def test_inline_schedule_unit_limit_and_count():
    """The Python unit count the step uses to choose the inline schedule agrees
    with the library's schedule sizing, and a call without a schedule buffer over
    256 work units is refused on the host before any pointer is touched."""
    import ctypes
    from deepseek_sparse_attention_mqa_gb300 import _abi
    L = _abi.lib()
    for args in [(64, 1, 64, 0, 64), (5, 3, 64, 0, 15), (1, 16384, 64, 0, 8192), (3, 4, 128, 2, 10),
                 (128, 2, 32, 0, 256), (7, 3, 16, 4, 19), (300, 1, 64, 0, 300)]:
        assert L.dsa_indexer_schedule_bytes(*args) == 32 + 32 * _abi.units_of(*args)
    fake = ctypes.c_void_p(0x1000)
    c = _abi.PagedCache()
    c.fmt, c.head_dim, c.page_kv, c.num_pages = 0, 128, 64, 2000
    c.values, c.scales, c.block_table = 0x1000, 0x2000, 0x3000
    c.val_page_stride, c.val_token_stride = 64 * 128, 128
    c.sc_page_stride, c.sc_token_stride = 256, 4
    c.bt_row_stride, c.max_pages_per_seq = 2000, 2000
    st = L.indexer_mqa_logits_paged(fake, None, 0, fake, 64, ctypes.byref(c), fake, 300, 1, 0, 300,
                                    None, 0, fake, 4096, 4096, None, None)
    assert st == _abi.DSA_ERR_CAPACITY


def test_noalloc_rejects_before_touching_the_fixed_array():
    """A call above 256 units with a bad argument is refused by the same host
    checks as the regular entry point, before the fixed array's address is
    looked up or its schedule build enqueued: with no GPU here, any CUDA call
    would have come back as DSA_ERR_CUDA instead."""
    L = _abi.lib()
    fake = ctypes.c_void_p(0x1000)
    c = _abi.PagedCache()
    c.fmt, c.head_dim, c.page_kv, c.num_pages = 0, 128, 64, 2000
    c.values, c.scales, c.block_table = 0x1000, 0x2000, 0x3000
    c.val_page_stride, c.val_token_stride = 64 * 128, 128
    c.sc_page_stride, c.sc_token_stride = 256, 4
    c.bt_row_stride, c.max_pages_per_seq = 2000, 2000
    call = lambda H, w, width: L.indexer_mqa_logits_paged_noalloc(
        fake, None, 0, w, H, ctypes.byref(c), fake, 300, 1, 0, 300, fake, 4096, width, None, None)
    assert call(48, fake, 4096) == _abi.DSA_ERR_UNSUPPORTED            # head count
    assert call(64, ctypes.c_void_p(0x1004), 4096) == _abi.DSA_ERR_INVALID_ARG  # misaligned weights
    assert call(64, fake, 8192) == _abi.DSA_ERR_INVALID_ARG            # row stride < width
