"""GPU parity of sparse MLA decode against the fp64 oracle (bf16 and FP8
latent caches, -1 padding, empty selections)."""
import numpy as np
import pytest
import torch

import oracle
import parity
from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.lib()
    oracle.build()


def random_indices(case, k, seed, pad_frac=0.0, empty_rows=()):
    rng = np.random.default_rng(seed)
    idx = np.full((case.rows, k), -1, np.int32)
    for r in range(case.rows):
        if r in empty_rows:
            continue
        vis = parity.visible(case, r)
        n = min(k, vis, int(round(k * (1 - pad_frac))))
        sel = rng.choice(vis, n, replace=False) if n else []
        slots = rng.choice(k, n, replace=False)
        idx[r, slots] = sel
    return idx


def run_mla(case, idx_np):
    dev = torch.device("cuda")
    lat = case.latent
    cache = _abi.make_cache(lat.fmt, lat.head_dim, lat.page_kv, lat.num_pages, lat.values,
                            lat.val_page_stride, lat.val_token_stride, lat.scales,
                            lat.sc_page_stride, lat.sc_token_stride, case.block_table)
    idx = torch.tensor(idx_np, device=dev)
    out = torch.full((case.rows, case.mla_heads, case.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((case.rows, case.mla_heads), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros((1,), dtype=torch.int32, device=dev)
    k = idx_np.shape[1]
    ws_n = _abi.mla_workspace_bytes(case.rows, case.mla_heads, case.d_qk, case.d_v, k)
    ws = torch.empty((max(ws_n, 16),), dtype=torch.uint8, device=dev)
    _abi.sparse_mla(case.q_mla, case.softmax_scale, cache, idx, k, out, lse, case.d_v,
                    None, case.next_n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse


def oracle_mla(case, idx_np, rows=None):
    cache, _ = parity.oracle_cache(case.latent, case.block_table)
    fmt = oracle.FMT_FP8 if case.latent.fmt == inputs.FMT_FP8 else oracle.FMT_BF16
    q = case.q_mla.cpu()
    if rows is None:
        return oracle.sparse_mla(q, case.softmax_scale, fmt, cache, idx_np, case.d_v,
                                 next_n=case.next_n)
    outs, lses = [], []
    for r in rows:
        o, l = oracle.sparse_mla(q[r:r + 1], case.softmax_scale, fmt, cache, idx_np[r:r + 1],
                                 case.d_v, seq_of_row=[r // case.next_n])
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


def test_tiny_bf16_latent():
    case = inputs.make_case("tiny", device="cuda")
    idx = random_indices(case, case.topk, 1, pad_frac=0.25)
    out, lse = run_mla(case, idx)
    ro, rl = oracle_mla(case, idx)
    parity.check_mla(out, lse, ro, rl)


def test_fp8_latent_576_512_with_empty_row():
    case = inputs.make_case("full_step", device="cuda", lens=[3000, 90, 2500], seed=31)
    idx = random_indices(case, 2048, 2, pad_frac=0.1, empty_rows=(1,))
    out, lse = run_mla(case, idx)
    ro, rl = oracle_mla(case, idx)
    parity.check_mla(out, lse, ro, rl)
    assert np.all(out[1].float().cpu().numpy() == 0) and np.all(np.isneginf(lse[1].cpu().numpy()))


@pytest.mark.parametrize("heads,d_qk,k,pad", [(128, 576, 2048, 0.0), (128, 576, 100, 0.3),
                                             (64, 576, 256, 0.0), (128, 512, 192, 0.1),
                                             (16, 576, 64, 0.5)])
def test_fp8_latent_shapes(heads, d_qk, k, pad):
    case = inputs.make_case("full_step", device="cuda", lens=[4000, 300, 64, 2500], seed=33,
                            mla=dict(heads=heads, d_qk=d_qk, d_v=512, fmt=inputs.FMT_FP8,
                                     scale=1.0 / np.sqrt(192)))
    idx = random_indices(case, k, 7, pad_frac=pad)
    out, lse = run_mla(case, idx)
    ro, rl = oracle_mla(case, idx)
    parity.check_mla(out, lse, ro, rl)


def test_fp8_latent_repeat_is_deterministic():
    case = inputs.make_case("full_step", device="cuda", lens=[3000, 2000], seed=34)
    idx = random_indices(case, 2048, 3)
    a = run_mla(case, idx)
    b = run_mla(case, idx)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_index_outside_the_block_table_sets_status_and_is_skipped():
    """A selected index past the sequence's block table, and one in a page the
    table leaves unused, are reported as DSA_DEV_BAD_INDEX and contribute
    nothing: the output equals the oracle's with those slots empty."""
    case = inputs.make_case("full_step", device="cuda", lens=[3000, 2500], seed=35)
    idx = random_indices(case, 256, 8)
    P = case.latent.page_kv
    max_pages = case.block_table.shape[1]
    bad = idx.copy()
    bad[0, 5] = max_pages * P + 10                      # beyond the table
    bad[1, 7] = 2500 + 2 * P                             # row 1 (2500 tokens): a page the table leaves unused
    assert int(case.block_table[1, (2500 + 2 * P) // P].item()) < 0
    dev = torch.device("cuda")
    lat = case.latent
    cache = _abi.make_cache(lat.fmt, lat.head_dim, lat.page_kv, lat.num_pages, lat.values,
                            lat.val_page_stride, lat.val_token_stride, lat.scales,
                            lat.sc_page_stride, lat.sc_token_stride, case.block_table)
    out = torch.full((case.rows, case.mla_heads, case.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((case.rows, case.mla_heads), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros((1,), dtype=torch.int32, device=dev)
    ws_n = _abi.mla_workspace_bytes(case.rows, case.mla_heads, case.d_qk, case.d_v, 256)
    ws = torch.empty((max(ws_n, 16),), dtype=torch.uint8, device=dev)
    _abi.sparse_mla(case.q_mla, case.softmax_scale, cache, torch.tensor(bad, device=dev), 256, out, lse,
                    case.d_v, None, case.next_n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) & _abi.DEV_BAD_INDEX
    expect = idx.copy()
    expect[0, 5] = -1
    expect[1, 7] = -1
    ro, rl = oracle_mla(case, expect)
    parity.check_mla(out, lse, ro, rl)
