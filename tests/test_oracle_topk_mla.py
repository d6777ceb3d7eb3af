"""Pins for the oracle's top-k and sparse MLA decode (CPU only).

Top-k: brute force on tiny rows, k >= visible length returns every visible
index, agreement with numpy's stable argsort / torch.topk when there are no ties.
Sparse MLA: top-k = every visible token equals dense softmax attention computed
by torch in fp64; one selected token gives out = V, lse = s; equal scores give
the mean of V and lse = s + ln n; permutations of the index list and -1 padding
change nothing.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_mqa_gb300 import inputs


# ------------------------------------------------------------------ top-k

def test_topk_brute_force_tiny(oracle):
    g = np.random.default_rng(1)
    for vis in range(0, 7):
        for k in range(1, 8):
            row = g.integers(-3, 4, size=8).astype(np.float64)   # many exact ties
            idx, cnt = oracle.topk(row[None, :], [vis], 1, k)
            take = min(k, vis)
            assert cnt[0] == take
            assert np.all(idx[0, take:] == -1)
            # brute force: the lexicographically best subset by (value desc, index asc)
            best = None
            for sub in itertools.combinations(range(vis), take):
                key = sorted(((-row[s], s) for s in sub))
                if best is None or key < best[0]:
                    best = (key, sub)
            want = [s for _, s in best[0]] if take else []
            assert list(idx[0, :take]) == want


def test_topk_k_at_least_visible_returns_all(oracle):
    row = np.random.default_rng(2).standard_normal((1, 40))
    for vis in (0, 1, 17, 40):
        idx, cnt = oracle.topk(row, [vis], 1, 64)
        assert cnt[0] == vis
        assert sorted(idx[0, :vis].tolist()) == list(range(vis))
        assert np.all(idx[0, vis:] == -1)


def test_topk_matches_numpy_and_torch_without_ties(oracle):
    g = np.random.default_rng(3)
    rows = g.standard_normal((6, 500))
    lens = [500, 300, 2, 77, 499, 128]
    idx, _ = oracle.topk(rows, lens, 1, 64)
    for r, L in enumerate(lens):
        want = np.argsort(-rows[r, :L], kind="stable")[:64]
        assert list(idx[r, :min(64, L)]) == list(want)
        tk = torch.topk(torch.tensor(rows[r, :L]), min(64, L)).indices.numpy()
        assert set(tk.tolist()) == set(idx[r, :min(64, L)].tolist())


def test_topk_next_n_windows(oracle):
    row = np.arange(10, dtype=np.float64)[None].repeat(3, 0)    # increasing logits
    idx, cnt = oracle.topk(row, [5], 3, 2)                       # vis = 3, 4, 5
    assert cnt.tolist() == [2, 2, 2]
    assert idx.tolist() == [[2, 1], [3, 2], [4, 3]]


# ------------------------------------------------------------- sparse MLA

def bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16)


def mla_cache(lat_vals, page_kv, perm, fmt, scales=None):
    """Single-sequence paged latent cache from logical rows [S, d] (already
    representable in the storage format)."""
    S, d = lat_vals.shape
    npg = (S + page_kv - 1) // page_kv
    bt = np.array([perm[:npg]], np.int32)
    pool = max(perm[:npg]) + 1
    if fmt == 2:
        row_bytes = 2 * d
        vals = np.zeros((pool, page_kv * row_bytes), np.uint8)
        b = lat_vals.to(torch.bfloat16).view(torch.uint8).numpy().reshape(S, row_bytes)
        scs = None
    else:
        row_bytes = d
        vals = np.full((pool, page_kv * row_bytes), 0x7F, np.uint8)
        b = lat_vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        scs = np.zeros((pool, page_kv * 4), np.uint8)
    for s in range(S):
        p, t = bt[0, s // page_kv], s % page_kv
        vals[p, t * row_bytes:(t + 1) * row_bytes] = b[s]
        if scs is not None:
            scs[p, t * 4:(t + 1) * 4] = np.frombuffer(np.float32(scales[s]).tobytes(), np.uint8)
    return dict(values=vals, val_page_stride=page_kv * row_bytes, val_token_stride=row_bytes,
                scales=scs, sc_page_stride=page_kv * 4, sc_token_stride=4, block_table=bt,
                page_kv=page_kv, num_pages=pool)


@pytest.mark.parametrize("fmt", [0, 2])
def test_mla_all_tokens_equals_dense_attention(oracle, fmt):
    g = torch.Generator().manual_seed(4)
    S, Hq, dqk, dv = 37, 5, 48, 32
    lat = torch.randn((S, dqk), generator=g)
    if fmt == 0:
        lat = lat.to(torch.float8_e4m3fn).to(torch.float32)
        sc = (torch.rand(S, generator=g) * 1.5 + 0.5)
    else:
        lat = lat.to(torch.bfloat16).to(torch.float32)
        sc = torch.ones(S)
    q = torch.randn((1, Hq, dqk), generator=g).to(torch.bfloat16)
    pc = mla_cache(lat, 16, [2, 0, 1], fmt, sc.numpy())
    cache = oracle.PagedBytes(**pc)
    idx = np.random.default_rng(0).permutation(S).astype(np.int32)[None]
    scale = 1 / math.sqrt(dqk)
    out, lse = oracle.sparse_mla(bf16_bits(q), scale, fmt, cache, idx, dv)
    C = lat.to(torch.float64) * sc.to(torch.float64)[:, None]
    Q = q.to(torch.float64)[0]
    logits = scale * Q @ C.T
    ref = torch.softmax(logits, dim=-1) @ C[:, :dv]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], torch.logsumexp(logits, -1).numpy(), rtol=1e-12)


def test_mla_single_token_and_equal_scores(oracle):
    g = torch.Generator().manual_seed(6)
    S, Hq, dqk, dv = 20, 3, 32, 16
    lat = torch.randn((S, dqk), generator=g).to(torch.bfloat16).to(torch.float32)
    cache = oracle.PagedBytes(**mla_cache(lat, 8, [0, 1, 2], 2))
    q = torch.randn((1, Hq, dqk), generator=g).to(torch.bfloat16)
    idx = np.full((1, 6), -1, np.int32)
    idx[0, 3] = 11
    out, lse = oracle.sparse_mla(bf16_bits(q), 0.25, 2, cache, idx, dv)
    C = lat.to(torch.float64)
    np.testing.assert_array_equal(out[0], C[11, :dv].expand(Hq, dv).numpy())
    np.testing.assert_allclose(lse[0], (0.25 * q.to(torch.float64)[0] @ C[11]).numpy(),
                               rtol=1e-14)
    # q = 0 -> every score is 0: out = mean of the selected V rows, lse = ln n
    sel = np.array([[1, 4, 9, 15, -1, 2]], np.int32)
    out, lse = oracle.sparse_mla(bf16_bits(torch.zeros((1, Hq, dqk))), 0.3, 2, cache, sel, dv)
    mean = C[[1, 4, 9, 15, 2], :dv].mean(0)
    np.testing.assert_allclose(out[0], mean.expand(Hq, dv).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(5), rtol=1e-14)
    # nothing selected: out = 0, lse = -inf
    out, lse = oracle.sparse_mla(bf16_bits(q), 0.3, 2, cache, np.full((1, 4), -1, np.int32), dv)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_mla_index_order_and_padding_invariance(oracle):
    case = inputs.make_case("tiny")
    lat = case.latent
    cache = oracle.PagedBytes(lat.values, lat.val_page_stride, lat.val_token_stride, None, 0, 0,
                              case.block_table, lat.page_kv, lat.num_pages)
    rng = np.random.default_rng(8)
    idx = np.stack([rng.choice(int(L), 40, replace=False) for L in case.context_lens]).astype(np.int32)
    a = oracle.sparse_mla(case.q_mla, case.softmax_scale, 2, cache, idx, case.d_v)
    perm = rng.permutation(40)
    padded = np.full((2, 64), -1, np.int32)
    padded[:, rng.choice(64, 40, replace=False)] = idx[:, perm]
    b = oracle.sparse_mla(case.q_mla, case.softmax_scale, 2, cache, padded, case.d_v)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13)
