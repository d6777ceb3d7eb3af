"""GPU parity of sparse MLA over a sliding window plus selected entries
(sparse_mla_decode_swa) against the fp64 oracle: one softmax over the first
topk_lens[r] entries of each row's index list in a compressed latent cache and
the last min(window, vis) visible tokens of a sliding-window cache, rows mapped
to sequences by cumulative query lengths.  Both MLA kernels are covered (the
tensor-core kernel at 576/512 and 512/512 FP8 with up to 128 heads, the
CUDA-core kernel at the bf16 80/64 shape), as are compressed caches that hold
two entries per physical block, empty and short histories, and rows with no
selected entry."""
import numpy as np
import pytest
import torch

import oracle
import parity
from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs
from oracle.cases import oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.lib()
    oracle.build()


def abi_cache(p, bt):
    return _abi.make_cache(p.fmt, p.head_dim, p.page_kv, p.num_pages, p.values, p.val_page_stride,
                           p.val_token_stride, p.scales, p.sc_page_stride, p.sc_token_stride, bt)


def run_case(c, use_window=True, use_tl=True, use_cum=True, next_n=1):
    dev = c.q.device
    out = torch.full((c.rows, c.heads, c.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((c.rows, c.heads), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    _abi.sparse_mla_swa(c.q, c.softmax_scale, abi_cache(c.sparse, c.sparse_bt), c.idx, c.k, out, lse, c.d_v,
                        topk_lens=c.topk_lens if use_tl else None,
                        swa=abi_cache(c.swa, c.swa_bt) if use_window else None,
                        window=c.window if use_window else 0, seq_lens=c.seq_lens,
                        cum_q=c.cum_q if use_cum else None, batch=c.batch, next_n=next_n, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sp, _ = oracle_cache(c.sparse, c.sparse_bt)
    sw, _ = oracle_cache(c.swa, c.swa_bt)
    ro, rl = oracle.sparse_mla_swa(c.q.cpu(), c.softmax_scale, c.fmt, sp, c.idx.cpu(), c.d_v, c.seq_lens.cpu(),
                                   c.topk_lens.cpu() if use_tl else None, sw if use_window else None,
                                   c.window if use_window else 0, c.cum_q.cpu() if use_cum else None, next_n)
    parity.check_mla(out, lse, ro, rl)
    return out, lse


@pytest.mark.parametrize("heads,d_qk,d_v", [(128, 576, 512), (64, 512, 512), (16, 576, 512)])
def test_tensor_core_shapes(heads, d_qk, d_v):
    c = inputs.make_swa_case(seed=heads + d_qk, device="cuda", seq_lens=(3000, 900, 130, 1, 0, 5000),
                             q_lens=(1, 3, 2, 1, 1, 2), heads=heads, d_qk=d_qk, d_v=d_v, k=256, window=128)
    run_case(c)


def test_cuda_core_bf16_shape():
    c = inputs.make_swa_case(seed=7, device="cuda", seq_lens=(200, 317, 64, 3), q_lens=(1, 2, 3, 2), heads=4,
                             d_qk=80, d_v=64, fmt=inputs.FMT_BF16, k=64, window=40, page_kv=32, swa_page_kv=32)
    run_case(c)


def test_full_size_rows_decode_shape():
    """The full decode step's MLA shape with a window: 128 heads, k 2048, window
    128, 64 single-token rows over contexts up to 131072 (a quarter of them in
    the compressed cache)."""
    g = torch.Generator().manual_seed(9)
    lens = torch.randint(8192, 131073, (64,), generator=g).tolist()
    c = inputs.make_swa_case(seed=9, device="cuda", seq_lens=lens, q_lens=[1] * 64, heads=128, k=2048,
                             window=128)
    run_case(c)


def test_two_entries_per_block_and_no_window():
    """A compressed cache holding 2 entries per physical block (page_kv 2, as a
    heavily compressed layer's view of 256-token blocks) read through the
    selected entries alone, with and without per-row lengths."""
    c = inputs.make_swa_case(seed=11, device="cuda", seq_lens=(4000, 700, 50), q_lens=(2, 1, 3), heads=32,
                             k=128, window=16, page_kv=2, ratio=128)
    run_case(c, use_window=False)
    run_case(c, use_window=False, use_tl=False)


def test_window_only_and_uniform_rows():
    c = inputs.make_swa_case(seed=12, device="cuda", seq_lens=(60, 1000, 2), q_lens=(2, 2, 2), heads=128,
                             k=64, window=300)
    c.topk_lens.zero_()                                  # window keys only
    run_case(c)
    run_case(c, use_cum=False, next_n=2)                 # the same rows without cumulative lengths


def test_plain_sparse_mla_unchanged_by_the_window_path():
    """sparse_mla_decode (no window, no lengths) and sparse_mla_decode_swa with
    neither give bit-identical outputs."""
    c = inputs.make_swa_case(seed=13, device="cuda", seq_lens=(900, 2000), q_lens=(1, 1), heads=128, k=512)
    out_a, lse_a = run_case(c, use_window=False, use_tl=False, use_cum=False, next_n=1)
    out_b = torch.empty_like(out_a)
    lse_b = torch.empty_like(lse_a)
    _abi.sparse_mla(c.q, c.softmax_scale, abi_cache(c.sparse, c.sparse_bt), c.idx, c.k, out_b, lse_b, c.d_v)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
