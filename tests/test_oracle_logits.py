"""Pins for the oracle's indexer logits (CPU only).

The oracle (plain C loops over the block table) is checked against: hand-worked
cases (tests/golden), a torch fp64 einsum on tensors dequantised by torch and
gathered through the block table by torch indexing, the special case that
reduces to a plain matrix-vector product, exact invariances (physical page
permutation, padded strides, positive homogeneity) and the FP8 <-> MXFP4
equivalence on values both formats represent exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_mqa_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP MX v1.0 magnitudes, codes 0..7


def paged_fp8(k_tokens, k_scale, page_kv, perm=None, val_pad=0, sc_pad=0, pool_extra=0):
    """Lay tokens [S, D] (float, exactly e4m3) and scales [S] out as a paged
    single-sequence cache.  Returns (oracle.PagedBytes-ready dict, block_table)."""
    S, D = k_tokens.shape
    npg = max(1, (S + page_kv - 1) // page_kv)
    pool = npg + pool_extra
    if perm is None:
        perm = list(range(pool))
    vstride = page_kv * D + val_pad
    sstride = page_kv * 4 + sc_pad
    vals = np.full((pool, vstride), 0x7F, np.uint8)
    scs = np.full((pool, sstride), 0xFF, np.uint8)
    kb = torch.tensor(k_tokens, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sb = np.asarray(k_scale, np.float32)
    bt = np.full((1, npg), -1, np.int32)
    for lp in range(npg):
        p = perm[lp]
        bt[0, lp] = p
        for t in range(page_kv):
            s = lp * page_kv + t
            if s < S:
                vals[p, t * D:(t + 1) * D] = kb[s]
                scs[p, t * 4:(t + 1) * 4] = np.frombuffer(sb[s:s + 1].tobytes(), np.uint8)
    return dict(values=vals, val_page_stride=vstride, val_token_stride=D, scales=scs,
                sc_page_stride=sstride, sc_token_stride=4, block_table=bt, page_kv=page_kv,
                num_pages=pool)


def e4m3_bytes(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def run_fp8(oracle, q, w, pc, ctx, next_n=1, **kw):
    cache = oracle.PagedBytes(**pc)
    return oracle.logits_fp8(q, w, cache, np.asarray(ctx, np.int32), next_n, **kw)


# ------------------------------------------------------------------ golden

def test_hand_worked_cases(oracle):
    with open(os.path.join(HERE, "golden", "indexer_hand_cases.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        q = e4m3_bytes(np.array(case["q"]))
        w = np.array(case["w"], np.float32)
        k = np.array(case["k"], np.float64)
        pc = paged_fp8(k, case["k_scale"], page_kv=1, perm=list(reversed(range(len(k)))))
        out = run_fp8(oracle, q, w, pc, [len(k)])
        assert np.array_equal(out, np.array(case["expect"])), case["name"]


# ------------------------------------------------- library cross-checks

def dense_reference_fp8(case):
    """torch fp64: dequantise with torch, gather logical tokens with torch
    indexing, einsum over (head, dim), relu, weight, scale."""
    kc = case.kcache
    P, D = case.page_kv, case.head_dim
    vals = kc.values[:, :P * D].reshape(kc.num_pages, P, D).contiguous()
    kv = vals.view(torch.float8_e4m3fn).to(torch.float64)
    ks = kc.scales[:, :P * 4].contiguous().view(torch.float32).reshape(kc.num_pages, P).to(torch.float64)
    q = case.q.view(torch.float8_e4m3fn).to(torch.float64)
    w = case.weights.to(torch.float64)
    outs = []
    for b in range(case.batch):
        L = int(case.context_lens[b])
        s = torch.arange(L)
        phys = case.block_table[b].long()[s // P]
        K = kv[phys, s % P]                    # [L, D]
        S = ks[phys, s % P]                    # [L]
        for i in range(case.next_n):
            r = b * case.next_n + i
            dots = torch.einsum("hd,sd->hs", q[r], K)
            outs.append((S * (w[r][:, None] * dots.clamp_min(0)).sum(0)).numpy())
    return outs


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("decode", dict(lens=[130, 64, 1, 0, 257])),
    ("decode", dict(lens=[50, 77], next_n=3, page_kv=32, num_heads=16, head_dim=64)),
    ("full_step", dict(lens=[129, 300], with_mla=False)),
])
def test_logits_match_torch_einsum(oracle, name, kw):
    case = inputs.make_case(name, **kw)
    kc = case.kcache
    cache = oracle.PagedBytes(kc.values, kc.val_page_stride, kc.val_token_stride, kc.scales,
                              kc.sc_page_stride, kc.sc_token_stride, case.block_table,
                              kc.page_kv, kc.num_pages)
    out = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, case.next_n,
                            width=case.width)
    ref = dense_reference_fp8(case)
    for r in range(case.rows):
        b, i = divmod(r, case.next_n)
        vis = oracle.visible(int(case.context_lens[b]), case.next_n, i)
        assert np.all(np.isnan(out[r, vis:]))          # never written past the window
        np.testing.assert_allclose(out[r, :vis], ref[r][:vis], rtol=1e-12, atol=1e-12)


def test_single_head_positive_reduces_to_matvec(oracle):
    g = torch.Generator().manual_seed(11)
    S, D = 70, 32
    # positive e4m3 values so that relu is the identity
    k = (torch.rand((S, D), generator=g) * 3 + 0.01).to(torch.float8_e4m3fn).to(torch.float64)
    q = (torch.rand((1, 1, D), generator=g) * 3 + 0.01).to(torch.float8_e4m3fn).to(torch.float64)
    pc = paged_fp8(k.numpy(), np.ones(S), page_kv=32, perm=[2, 0, 1])
    out = run_fp8(oracle, e4m3_bytes(q.numpy()), np.ones((1, 1), np.float32), pc, [S])
    np.testing.assert_allclose(out[0], k.numpy() @ q[0, 0].numpy(), rtol=1e-13)


# ------------------------------------------------------------ invariances

def test_page_permutation_and_padding_invariance(oracle):
    g = torch.Generator().manual_seed(5)
    S, D, H = 150, 64, 8
    k = torch.randn((S, D), generator=g).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    sc = (torch.rand(S, generator=g) * 1.5 + 0.5).numpy()
    q = e4m3_bytes(torch.randn((2, H, D), generator=g).numpy())
    w = (torch.randn((2, H), generator=g) / 3).numpy().astype(np.float32)
    a = run_fp8(oracle, q, w, paged_fp8(k, sc, 32), [S, S][:1] * 1, next_n=2)
    b = run_fp8(oracle, q, w, paged_fp8(k, sc, 32, perm=[6, 2, 0, 5, 1, 3, 4], val_pad=48,
                                        sc_pad=16, pool_extra=2), [S], next_n=2)
    assert np.array_equal(np.nan_to_num(a, nan=7.0), np.nan_to_num(b, nan=7.0))


def test_positive_homogeneity(oracle):
    case = inputs.make_case("decode", lens=[100, 200], num_heads=8, head_dim=32)
    kc = case.kcache
    cache = oracle.PagedBytes(kc.values, kc.val_page_stride, kc.val_token_stride, kc.scales,
                              kc.sc_page_stride, kc.sc_token_stride, case.block_table,
                              kc.page_kv, kc.num_pages)
    a = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 1)
    b = oracle.logits_fp8(case.q, case.weights * 2, cache, case.context_lens, 1)
    ok = ~np.isnan(a)
    assert np.array_equal(b[ok], 2 * a[ok])


def test_heads_add_up(oracle):
    case = inputs.make_case("decode", lens=[90], num_heads=6, head_dim=32)
    kc = case.kcache
    cache = oracle.PagedBytes(kc.values, kc.val_page_stride, kc.val_token_stride, kc.scales,
                              kc.sc_page_stride, kc.sc_token_stride, case.block_table,
                              kc.page_kv, kc.num_pages)
    full = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 1)
    parts = sum(oracle.logits_fp8(case.q[:, h:h + 1].contiguous(),
                                  case.weights[:, h:h + 1].contiguous(), cache,
                                  case.context_lens, 1) for h in range(6))
    np.testing.assert_allclose(full, parts, rtol=1e-12, atol=1e-12)


def test_row_range_selects_rows(oracle):
    case = inputs.make_case("decode", lens=[40, 70, 10], next_n=2, num_heads=4, head_dim=32)
    kc = case.kcache
    cache = oracle.PagedBytes(kc.values, kc.val_page_stride, kc.val_token_stride, kc.scales,
                              kc.sc_page_stride, kc.sc_token_stride, case.block_table,
                              kc.page_kv, kc.num_pages)
    full = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 2, width=70)
    part = oracle.logits_fp8(case.q, case.weights, cache, case.context_lens, 2, row_begin=2,
                             row_end=5, width=70)
    assert np.array_equal(np.nan_to_num(full[2:5], nan=3.0), np.nan_to_num(part, nan=3.0))


# ------------------------------------------------------------------ MXFP4

def unpack_mxfp4(packed, scales):
    """Test-side decode from the OCP value grid and torch's ue8m0 conversion."""
    p = torch.as_tensor(packed)
    nib = torch.stack([p & 0xF, p >> 4], dim=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    grid = torch.tensor(E2M1_GRID, dtype=torch.float64)
    mag = grid[(nib & 7).long()]
    val = torch.where((nib & 8) > 0, -mag, mag)
    sc = torch.as_tensor(scales).contiguous().view(torch.float8_e8m0fnu).to(torch.float64)
    return val * sc.repeat_interleave(32, dim=-1)


def test_mxfp4_logits_match_torch_einsum(oracle):
    case = inputs.make_case("spec_mxfp4", lens=[0, 1, 33, 95, 64], val_pad=1024, sc_pad=64)
    kc = case.kcache
    P, D = case.page_kv, case.head_dim
    cache = oracle.PagedBytes(kc.values, kc.val_page_stride, kc.val_token_stride, kc.scales,
                              kc.sc_page_stride, kc.sc_token_stride, case.block_table,
                              kc.page_kv, kc.num_pages)
    out = oracle.logits_mxfp4(case.q, case.q_scales, case.weights, cache, case.context_lens,
                              case.next_n, width=96)
    kvals = unpack_mxfp4(kc.values[:, :P * D // 2].reshape(kc.num_pages, P, D // 2),
                         kc.scales[:, :P * D // 32].reshape(kc.num_pages, P, D // 32))
    q = unpack_mxfp4(case.q, case.q_scales)
    w = case.weights.to(torch.float64)
    for b in range(case.batch):
        L = int(case.context_lens[b])
        s = torch.arange(L)
        K = kvals[case.block_table[b].long()[s // P], s % P]
        for i in range(case.next_n):
            r = b * case.next_n + i
            vis = oracle.visible(L, case.next_n, i)
            ref = (w[r][:, None] * torch.einsum("hd,sd->hs", q[r], K).clamp_min(0)).sum(0)
            np.testing.assert_allclose(out[r, :vis], ref[:vis].numpy(), rtol=1e-12, atol=1e-12)
            assert np.all(np.isnan(out[r, vis:]))


def test_mxfp4_equals_fp8_on_shared_values(oracle):
    """Values on the e2m1 grid with unit block scales are exact in e4m3 too; the
    two oracle entry points must then agree bit for bit."""
    g = torch.Generator().manual_seed(9)
    S, D, H = 45, 64, 3
    kcode = torch.randint(0, 16, (S, D), generator=g)
    qcode = torch.randint(0, 16, (1, H, D), generator=g)
    grid = torch.tensor(E2M1_GRID, dtype=torch.float64)

    def val(c):
        m = grid[(c & 7)]
        return torch.where((c & 8) > 0, -m, m)

    def pack(c):
        return (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8).numpy()

    P = 32
    npg = (S + P - 1) // P
    vals = np.full((npg, P * D // 2), 0x7F, np.uint8)
    scs = np.full((npg, P * 2), 0xFF, np.uint8)
    kp = pack(kcode)
    for s in range(S):
        vals[s // P, (s % P) * 32:(s % P + 1) * 32] = kp[s]
        scs[s // P, (s % P) * 2:(s % P + 1) * 2] = 127
    bt = np.arange(npg, dtype=np.int32)[None]
    mx = oracle.PagedBytes(vals, P * 32, 32, scs, P * 2, 2, bt, P, npg)
    w = np.array([[0.5, -1.0, 2.0]], np.float32)
    a = oracle.logits_mxfp4(pack(qcode), np.full((1, H, 2), 127, np.uint8), w, mx, [S], 1)
    pc = paged_fp8(val(kcode).numpy(), np.ones(S), P)
    b = run_fp8(oracle, e4m3_bytes(val(qcode).numpy()), w, pc, [S])
    assert np.array_equal(a, b)
