"""GPU parity of the K-cache quantise/scatter (dsa_kv_quantize_scatter) against
the oracle, byte for byte: the whole value and scale buffers after the scatter,
from the same initial contents, must be identical (codes, scales, and every byte
that no slot addresses left as it was)."""
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


def new_k(n, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((n, D), generator=g)
    if n >= 6:
        k[0] = 0.0                                     # all-zero row
        k[1] *= 1e-30                                  # subnormal-range inputs
        k[2] *= 3e4                                    # large magnitudes
        k[3, ::2] = -0.0                               # signed zeros
        k[4, : D // 2] = 0.0                           # a zero half (zero MX blocks)
        k[5] = torch.round(k[5] * 8) / 8               # exactly representable values
    return k.to(dtype)


def run_case(fmt, D, P, pages, n, dtype, seed, vpad=0, spad=0, skip_every=7):
    dev = torch.device("cuda")
    tok = D if fmt == 0 else D // 2
    stok = 4 if fmt == 0 else D // 32
    vps, sps = P * tok + vpad, P * stok + spad
    init_v = torch.randint(0, 256, (pages, vps), generator=torch.Generator().manual_seed(seed + 1),
                           dtype=torch.uint8)
    init_s = torch.randint(0, 256, (pages, sps), generator=torch.Generator().manual_seed(seed + 2),
                           dtype=torch.uint8)
    k = new_k(n, D, dtype, seed)
    rng = np.random.default_rng(seed)
    slots = rng.permutation(pages * P)[:n].astype(np.int64)
    if skip_every:
        slots[::skip_every] = -1                        # padding tokens
    vals, scs = init_v.to(dev), init_s.to(dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    cache = _abi.make_cache(fmt, D, P, pages, vals, vps, tok, scs, sps, stok, bt)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    _abi.kv_quantize_scatter(k.to(dev), torch.from_numpy(slots).to(dev), cache, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.PagedBytes(init_v.numpy().copy(), vps, tok, init_s.numpy().copy(), sps, stok,
                            np.zeros((1, 1), np.int32), P, pages)
    oracle.quantize_scatter(k, slots, fmt, ref)
    gv, gs = vals.cpu().numpy().reshape(-1), scs.cpu().numpy().reshape(-1)
    bad_v = np.nonzero(gv != ref.values)[0]
    bad_s = np.nonzero(gs != ref.scales)[0]
    assert bad_v.size == 0, "value bytes differ at %s" % bad_v[:8]
    assert bad_s.size == 0, "scale bytes differ at %s" % bad_s[:8]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,P,n,vpad,spad", [
    (128, 64, 1, 0, 0),
    (128, 64, 257, 0, 0),            # several CTAs and a ragged tail
    (32, 32, 100, 16, 16),           # padded strides
    (64, 64, 3000, 0, 0),
    (576, 64, 130, 0, 0),            # the MLA latent row (512 + 64)
])
def test_fp8_scatter_bit_exact(dtype, D, P, n, vpad, spad):
    run_case(0, D, P, max(4, -(-n // P) * 2), n, dtype, seed=D + n, vpad=vpad, spad=spad)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,P,n,vpad,spad", [
    (64, 32, 1, 0, 0),
    (64, 32, 500, 1024, 64),         # the speculative workload's padded layout
    (128, 64, 257, 0, 0),
    (256, 64, 77, 32, 16),           # more than one pass of 32 chunks
    (512, 32, 40, 0, 0),
])
def test_mxfp4_scatter_bit_exact(dtype, D, P, n, vpad, spad):
    run_case(1, D, P, max(4, -(-n // P) * 2), n, dtype, seed=3 * D + n, vpad=vpad, spad=spad)


def test_empty_and_bad_slot():
    dev = torch.device("cuda")
    D, P, pages = 64, 32, 2
    vals = torch.zeros((pages, P * D), dtype=torch.uint8, device=dev)
    scs = torch.zeros((pages, P * 4), dtype=torch.uint8, device=dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    cache = _abi.make_cache(0, D, P, pages, vals, P * D, D, scs, P * 4, 4, bt)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    k = torch.randn((2, D), device=dev)
    _abi.kv_quantize_scatter(k[:0], torch.zeros((0,), dtype=torch.int64, device=dev), cache, status)
    _abi.kv_quantize_scatter(k, torch.tensor([3, pages * P + 5], dtype=torch.int64, device=dev), cache, status)
    torch.cuda.synchronize()
    assert _abi.device_status(status) & _abi.DEV_BAD_PAGE
    assert int(vals[0, 3 * D:4 * D].ne(0).sum()) > 0            # the good token was written


def test_scattered_cache_feeds_the_indexer():
    """New K written by the scatter into an indexer cache is what the logits
    kernel then scores: the logits over the GPU-scattered cache match the
    oracle's logits over the oracle-scattered cache (same bytes)."""
    dev = torch.device("cuda")
    case = inputs.make_case("decode", device=dev, lens=[700, 129, 64], num_heads=32, head_dim=64,
                            page_kv=32, width=704, seed=31, with_mla=False)
    kc = case.kcache
    # rewrite every token of every sequence through the scatter
    bt = case.block_table.cpu().numpy()
    slots = []
    for b, L in enumerate(case.context_lens.cpu().tolist()):
        slots += [int(bt[b, s // kc.page_kv]) * kc.page_kv + s % kc.page_kv for s in range(L)]
    k = torch.randn((len(slots), kc.head_dim), generator=torch.Generator().manual_seed(32)).to(torch.bfloat16)
    # the oracle scatters the same rows into a copy of the cache as it was before
    before, _ = parity.oracle_cache(kc, case.block_table)
    ref_cache = oracle.PagedBytes(before.values.copy(), before.vps, before.vts, before.scales.copy(), before.sps,
                                  before.sts, before.block_table, before.page_kv, before.num_pages)
    oracle.quantize_scatter(k, slots, 0, ref_cache)
    st = SparseAttentionStep(case, with_mla=False)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    _abi.kv_quantize_scatter(k.to(dev), torch.tensor(slots, dtype=torch.int64, device=dev), st.kcache, status)
    st.logits.fill_(float("nan"))
    st.run()
    torch.cuda.synchronize()
    assert _abi.device_status(status) == 0 and st.device_status() == 0
    assert np.array_equal(ref_cache.values, kc.values.cpu().numpy().reshape(-1))
    assert np.array_equal(ref_cache.scales, kc.scales.cpu().numpy().reshape(-1))
    ref = oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), ref_cache, case.context_lens.cpu(), 1,
                            width=case.width)
    vis = [parity.visible(case, r) for r in range(case.rows)]
    parity.check_logits(list(st.logits.cpu().numpy()), list(ref), vis)
