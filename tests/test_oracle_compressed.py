"""Pins of the oracle over a compressed indexer K cache (CPU): a row that sees
vis tokens sees floor(vis / ratio) entries.  Checked against hand-enumerated
windows, against the uncompressed oracle on the truncated context (decode
rows), against torch fp64 einsum over the entries each draft row sees, and the
top-k over those entries only."""
import numpy as np
import torch

import oracle
from deepseek_sparse_attention_mqa_gb300 import inputs
from oracle.cases import oracle_cache


def test_visible_entries_hand_enumerated():
    # L = 13 tokens, next_n = 3 draft rows, ratio 4: windows 11, 12, 13 tokens
    assert [oracle.visible(13, 3, i, 4) for i in range(3)] == [2, 3, 3]
    assert [oracle.visible(13, 3, i) for i in range(3)] == [11, 12, 13]
    assert [oracle.visible(3, 3, i, 2) for i in range(3)] == [0, 1, 1]
    assert oracle.visible(0, 1, 0, 4) == 0 and oracle.visible(7, 1, 0, 8) == 0


def test_decode_rows_equal_truncated_context():
    case = inputs.make_case("decode", lens=[64, 257, 1000, 3], num_heads=8, head_dim=32, width=1000, seed=3)
    cache, _ = oracle_cache(case.kcache, case.block_table)
    for ratio in (2, 4, 128):
        a = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 1, width=1000, ratio=ratio)
        trunc = case.context_lens // ratio
        b = oracle.logits_fp8(case.q, case.weights, cache, trunc, 1, width=1000)
        for r in range(case.rows):
            v = int(trunc[r])
            assert np.array_equal(a[r, :v], b[r, :v])
            assert np.all(np.isnan(a[r, v:]))


def test_draft_rows_against_einsum():
    case = inputs.make_case("decode", lens=[130, 40], next_n=3, num_heads=4, head_dim=32, page_kv=32,
                            width=200, seed=4)
    cache, _ = oracle_cache(case.kcache, case.block_table)
    ratio = 4
    lg = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 3, width=200, ratio=ratio)
    qf = case.q.view(torch.float8_e4m3fn).double()
    P, D = case.page_kv, case.head_dim
    for r in range(case.rows):
        b, i = divmod(r, 3)
        L = int(case.context_lens[b])
        vis = max(0, min(L - 3 + i + 1, L)) // ratio
        rows = []
        for s in range(vis):
            pg = int(case.block_table[b, s // P])
            raw = case.kcache.values[pg, (s % P) * D:(s % P) * D + D].view(torch.float8_e4m3fn).double()
            sc = case.kcache.scales[pg, (s % P) * 4:(s % P) * 4 + 4].view(torch.float32).double()
            rows.append((raw, sc))
        for s, (k, sc) in enumerate(rows):
            dots = torch.relu(qf[r] @ k)                       # [H]
            want = float(sc) * float((case.weights[r].double() * dots).sum())
            assert abs(lg[r, s] - want) <= 1e-12 * max(1.0, abs(want))
        assert np.all(np.isnan(lg[r, vis:]))


def test_topk_over_visible_entries_only():
    g = torch.Generator().manual_seed(5)
    lens = [100, 9, 0, 41]
    lg = torch.randn((4, 100), generator=g).double().numpy()
    idx, cnt = oracle.topk(lg, lens, 1, 8, ratio=4)
    for r, L in enumerate(lens):
        v = L // 4
        assert cnt[r] == min(8, v)
        want = sorted(np.argsort(-lg[r, :v], kind="stable")[:min(8, v)].tolist())
        assert sorted(idx[r, :cnt[r]].tolist()) == want and np.all(idx[r, cnt[r]:] == -1)
