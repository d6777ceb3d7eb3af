"""GPU parity of the indexer over compressed K caches against the oracle: a
row that sees vis tokens scores floor(vis / ratio) cache entries (the CSA
index length context_len // 4), and layers of different compression ratios
share one block table and physical pool, each with its own page size (a
64-token storage block holding 64 entries of a ratio-1 layer and 32 states of
a ratio-2 layer).  Logits element by element, entries past each row's window
untouched, and top-k under the tolerance rule; also through the prebuilt
schedule and the fused score + top-k launch."""
import dataclasses

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


def check_case(case, fused=False, inline_schedule=None):
    st = SparseAttentionStep(case, with_mla=False, fused=fused, inline_schedule=inline_schedule)
    st.logits.fill_(float("nan"))
    st.idx.fill_(-7)
    st.run()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    cache, _ = parity.oracle_cache(case.kcache, case.block_table)
    ctx = case.context_lens.cpu()
    if case.fmt == inputs.FMT_FP8:
        ref = oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), cache, ctx, case.next_n, width=case.width,
                                ratio=case.ratio)
    else:
        ref = oracle.logits_mxfp4(case.q.cpu(), case.q_scales.cpu(), case.weights.cpu(), cache, ctx,
                                  case.next_n, width=case.width, ratio=case.ratio)
    vis = [parity.visible(case, r) for r in range(case.rows)]
    g = st.logits.cpu().numpy()
    parity.check_logits(list(g), list(ref), vis)
    for r, v in enumerate(vis):
        assert np.all(np.isnan(g[r][v:])), "row %d written past its entries" % r
    scale = max([float(np.max(np.abs(ref[r, :v]))) for r, v in enumerate(vis) if v] + [1.0])
    parity.check_topk_tolerant(st.idx.cpu().numpy(), ref, vis, case.topk, scale)
    counts = st.count.cpu().numpy()
    assert list(counts) == [min(v, case.topk) for v in vis]


@pytest.mark.parametrize("fused", [False, True])
def test_csa_ratio4_decode(fused):
    case = inputs.make_case("decode", device="cuda", lens=[0, 3, 4, 5, 400, 8191, 30000, 127],
                            num_heads=64, head_dim=128, topk=512, ratio=4, width=0, seed=61)
    assert case.width == 30000 // 4
    check_case(case, fused=fused)


def test_ratio2_draft_rows_page32():
    case = inputs.make_case("decode", device="cuda", lens=[1, 2, 63, 64, 65, 1000, 2049], next_n=3,
                            num_heads=16, head_dim=64, page_kv=32, topk=128, ratio=2, width=0, seed=62)
    check_case(case)


def test_mxfp4_ratio4():
    case = inputs.make_case("spec_mxfp4", device="cuda", batch=40, ratio=4, seed=63)
    check_case(case)


def test_ratio4_prebuilt_schedule():
    # 300 sequences: above the inline-schedule limit, so the schedule kernel
    # computes the compressed windows
    case = inputs.make_case("decode", device="cuda", lens=[(i * 97) % 3000 for i in range(300)],
                            num_heads=32, head_dim=64, topk=64, ratio=4, width=0, seed=64)
    check_case(case)


def test_layers_of_two_ratios_share_the_block_table():
    """One block table over 64-token storage blocks: the ratio-1 layer's cache
    has 64 entries per page, the ratio-2 layer's 32 states per page of the same
    physical block ids."""
    a = inputs.make_case("decode", device="cuda", lens=[70, 640, 3000, 1], num_heads=32, head_dim=64,
                         page_kv=64, topk=256, seed=65)
    g = torch.Generator(device="cuda").manual_seed(66)
    pool, D = a.kcache.num_pages, a.head_dim
    vals = inputs._to_e4m3_bytes(torch.randn((pool, 32 * D), generator=g, device="cuda"))
    scs = (torch.rand((pool, 32), generator=g, device="cuda") * 1.5 + 0.5).contiguous().view(torch.uint8)
    kc2 = inputs.Paged(inputs.FMT_FP8, D, 32, pool, vals.reshape(pool, 32 * D).contiguous(), 32 * D, D,
                       scs.reshape(pool, 128), 128, 4)
    b = dataclasses.replace(a, kcache=kc2, ratio=2, width=3000 // 2)
    check_case(a)
    check_case(b)
