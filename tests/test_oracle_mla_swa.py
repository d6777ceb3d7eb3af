"""Pins of the oracle's sparse MLA over a sliding window plus selected entries
(CPU): against softmax attention computed densely by torch in fp64 over the
keys gathered and dequantised by torch (e4m3 and bf16 through torch's own
conversions); the per-row top-k length as truncation of the index row; the
cumulative query lengths as the uniform next_n layout when they are uniform."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_mqa_gb300 import inputs
from oracle.cases import oracle_cache


def torch_rows(p: inputs.Paged, bt, b, positions):
    """Latent rows (fp64 [n, D]) of logical positions of sequence b, decoded by torch."""
    P, D = p.page_kv, p.head_dim
    out = []
    for s in positions:
        pg = int(bt[b, s // P])
        if p.fmt == inputs.FMT_FP8:
            raw = p.values[pg, (s % P) * D:(s % P) * D + D]
            v = raw.view(torch.float8_e4m3fn).double()
            sc = p.scales[pg, (s % P) * 4:(s % P) * 4 + 4].view(torch.float32).double()
            out.append(v * sc)
        else:
            raw = p.values[pg, (s % P) * 2 * D:(s % P) * 2 * D + 2 * D]
            out.append(raw.view(torch.bfloat16).double())
    return torch.stack(out) if out else torch.zeros((0, D), dtype=torch.float64)


def dense_reference(c: inputs.SwaCase, use_window=True, use_tl=True):
    out = torch.zeros((c.rows, c.heads, c.d_v), dtype=torch.float64)
    lse = torch.full((c.rows, c.heads), -math.inf, dtype=torch.float64)
    cum = c.cum_q.tolist()
    for b in range(c.batch):
        ql = cum[b + 1] - cum[b]
        L = int(c.seq_lens[b])
        for i in range(ql):
            r = cum[b] + i
            vis = max(0, min(L - ql + i + 1, L))
            kr = min(c.k, max(0, int(c.topk_lens[r]))) if use_tl else c.k
            sel = [int(s) for s in c.idx[r, :kr].tolist() if s >= 0]
            keys = [torch_rows(c.sparse, c.sparse_bt, b, sel)]
            if use_window:
                w = min(c.window, vis)
                keys.append(torch_rows(c.swa, c.swa_bt, b, list(range(vis - w, vis))))
            K = torch.cat(keys)
            if K.shape[0] == 0:
                continue
            qd = c.q[r].double()
            s = (qd @ K[:, :c.d_qk].T) * c.softmax_scale
            lse[r] = torch.logsumexp(s, dim=1)
            out[r] = torch.softmax(s, dim=1) @ K[:, :c.d_v]
    return out.numpy(), lse.numpy()


def run_oracle(c, use_window=True, use_tl=True, cum=True, next_n=1):
    sp, _ = oracle_cache(c.sparse, c.sparse_bt)
    sw, _ = oracle_cache(c.swa, c.swa_bt)
    return oracle.sparse_mla_swa(c.q, c.softmax_scale, c.fmt, sp, c.idx, c.d_v, c.seq_lens,
                                 c.topk_lens if use_tl else None, sw if use_window else None,
                                 c.window if use_window else 0, c.cum_q if cum else None, next_n)


@pytest.mark.parametrize("fmt,d_qk,d_v", [(inputs.FMT_FP8, 576, 512), (inputs.FMT_BF16, 80, 64),
                                          (inputs.FMT_FP8, 512, 512)])
def test_dense_torch_reference(fmt, d_qk, d_v):
    c = inputs.make_swa_case(seed=3, seq_lens=(300, 1000, 70, 5), q_lens=(1, 3, 2, 4), heads=4, d_qk=d_qk,
                             d_v=d_v, fmt=fmt, k=40, window=50, page_kv=32, swa_page_kv=64)
    o, l = run_oracle(c)
    ro, rl = dense_reference(c)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.max(np.abs(o - ro)) < 1e-10
    assert np.max(np.abs(l[fin] - rl[fin])) < 1e-10


def test_window_covers_short_sequences_and_empty_rows():
    # window longer than the history: every visible token; a row with no key
    c = inputs.make_swa_case(seed=4, seq_lens=(3, 0, 40), q_lens=(2, 1, 1), heads=2, d_qk=80, d_v=64,
                             fmt=inputs.FMT_BF16, k=8, window=100)
    c.topk_lens[:] = 0                                  # window keys only
    o, l = run_oracle(c)
    ro, rl = dense_reference(c)
    assert np.all(np.isneginf(l[2])) and np.all(o[2] == 0)   # sequence of length 0: no key
    fin = np.isfinite(rl)
    assert np.max(np.abs(o - ro)) < 1e-10 and np.max(np.abs(l[fin] - rl[fin])) < 1e-10


def test_topk_lens_is_truncation():
    c = inputs.make_swa_case(seed=5, heads=4, k=64, window=0)
    o, l = run_oracle(c, use_window=False)
    idx = c.idx.clone()
    for r in range(c.rows):
        idx[r, int(c.topk_lens[r]):] = -1
    sp, _ = oracle_cache(c.sparse, c.sparse_bt)
    seq_of_row = [b for b in range(c.batch) for _ in range(int(c.cum_q[b + 1] - c.cum_q[b]))]
    o2, l2 = oracle.sparse_mla(c.q, c.softmax_scale, c.fmt, sp, idx, c.d_v, seq_of_row=seq_of_row)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_uniform_cum_q_equals_next_n():
    c = inputs.make_swa_case(seed=6, seq_lens=(200, 90, 500), q_lens=(2, 2, 2), heads=2, k=16, window=30)
    a = run_oracle(c, cum=True)
    b = run_oracle(c, cum=False, next_n=2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
