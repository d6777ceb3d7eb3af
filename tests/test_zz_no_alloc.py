"""The allocation-free indexer entry point, indexer_mqa_logits_paged_noalloc.

It serves callers of this library that cannot allocate device memory -- a
plugin living under a host framework that owns the device allocator, or a
serving path that must not call cudaMalloc while handling requests -- by keeping
the indexer schedule in a fixed array inside the library instead of a
caller-owned buffer.  Its logits must agree with those of the regular entry
point (which takes a caller-allocated schedule) within the logits tolerance, on
two calls in a row: the fixed array keeps the previous call's schedule, and the
second call, with other lengths, must not be affected by it.

This file is collected last on purpose, and passes alone in a fresh process or
after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parity
from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs
from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.lib()
    oracle.build()


def regular_logits(case):
    """Logits through indexer_mqa_logits_paged with a caller-allocated schedule."""
    st = SparseAttentionStep(case, with_mla=False)
    st.logits.fill_(float("nan"))
    st.indexer_chunk(0, case.rows)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    return st.logits.cpu().numpy(), st


def noalloc_logits(case, st):
    """Same call through the allocation-free entry point (no schedule buffer)."""
    out = torch.full_like(st.logits, float("nan"))
    status = torch.zeros((1,), dtype=torch.int32, device=out.device)
    _abi.mqa_logits_noalloc(case.q, case.q_scales, case.fmt, case.weights, case.num_heads,
                            st.kcache, case.context_lens, case.batch, case.next_n, 0, case.rows,
                            out, st.width, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.cpu().numpy()


def check_same(case, ref, got):
    vis = [parity.visible(case, r) for r in range(case.rows)]
    parity.check_logits(list(got), list(ref), vis)
    for r, v in enumerate(vis):
        assert np.all(np.isnan(got[r][v:])), "row %d written past its visible length" % r


def test_two_calls_in_a_row_match_the_regular_entry_point():
    # first call: 9 sequences with long contexts; second call: 4 short ones, so a
    # stale schedule from the first call would send the second one wrong
    first = inputs.make_case("decode", device="cuda", lens=[4000, 17, 0, 2500, 129, 3333, 64, 1, 900],
                             width=4096, seed=71)
    second = inputs.make_case("decode", device="cuda", lens=[300, 5, 1000, 64], next_n=2,
                              num_heads=32, head_dim=64, page_kv=32, width=1024, seed=72)
    for case in (first, second):
        ref, st = regular_logits(case)
        got = noalloc_logits(case, st)
        check_same(case, ref, got)


def test_over_256_units_use_the_fixed_array():
    # 300 sequences: more units than the logits kernel builds itself, so the
    # schedule goes through the library's fixed array; then a small call (inline
    # schedule) and the large one again
    big = inputs.make_case("decode", device="cuda", lens=[(i * 37) % 600 + 1 for i in range(300)], width=640,
                           seed=74)
    small = inputs.make_case("decode", device="cuda", lens=[700, 3], width=704, seed=75)
    assert _abi.units_of(big.batch, big.next_n, big.num_heads, 0, big.rows) > _abi.INLINE_UNITS
    for case in (big, small, big):
        ref, st = regular_logits(case)
        check_same(case, ref, noalloc_logits(case, st))


def check_oracle(case, got):
    """The allocation-free call's logits against the fp64 oracle."""
    cache, _ = parity.oracle_cache(case.kcache, case.block_table)
    ref = oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), cache, case.context_lens.cpu(),
                            case.next_n, width=case.width)
    vis = [parity.visible(case, r) for r in range(case.rows)]
    parity.check_logits(list(got), list(ref), vis)


def test_fixed_array_rebuilt_when_the_call_changes():
    # three calls above 256 units back to back, all through the fixed array: 300
    # sequences, then 400 shorter ones with next_n 2 and another head count (so
    # other unit sizes and tile counts), then the first call again.  A schedule
    # left over from the previous call (skipped or partly rebuilt) would send
    # each call's work to the wrong rows and tokens.
    a = inputs.make_case("decode", device="cuda", lens=[(i * 37) % 600 + 1 for i in range(300)],
                         num_heads=16, head_dim=64, width=640, seed=76)
    b = inputs.make_case("decode", device="cuda", lens=[(i * 13) % 150 for i in range(400)],
                         next_n=2, num_heads=32, head_dim=64, page_kv=32, width=160, seed=77)
    for case in (a, b):
        assert _abi.units_of(case.batch, case.next_n, case.num_heads, 0, case.rows) > _abi.INLINE_UNITS
    for case in (a, b, a):
        ref, st = regular_logits(case)
        got = noalloc_logits(case, st)
        check_same(case, ref, got)
        check_oracle(case, got)


def test_mxfp4_through_the_noalloc_entry_point():
    case = inputs.make_case("spec_mxfp4", device="cuda", lens=[0, 1, 33, 700, 64, 2049],
                            width=2048 + 64, seed=73)
    ref, st = regular_logits(case)
    for _ in range(2):
        check_same(case, ref, noalloc_logits(case, st))


def test_too_many_work_units_is_refused():
    # 70000 prefill rows at 64 heads = 17500 units > 8191: refused on the host,
    # before any pointer is touched
    L = _abi.lib()
    fake = ctypes.c_void_p(0x1000)
    c = _abi.PagedCache()
    c.fmt, c.head_dim, c.page_kv, c.num_pages = 0, 128, 64, 2000
    c.values, c.scales, c.block_table = 0x1000, 0x2000, 0x3000
    c.val_page_stride, c.val_token_stride = 64 * 128, 128
    c.sc_page_stride, c.sc_token_stride = 256, 4
    c.bt_row_stride, c.max_pages_per_seq = 2000, 2000
    st = L.indexer_mqa_logits_paged_noalloc(fake, None, 0, fake, 64, ctypes.byref(c), fake, 1, 70000,
                                            0, 70000, fake, 70000, 70000, None, None)
    assert st == _abi.DSA_ERR_CAPACITY
