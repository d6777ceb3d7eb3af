"""Pins of the oracle's K-cache quantise/scatter (CPU).

The encoders are pinned to the formats by brute force (the nearest of all
codes, ties to the even code, found by search over the decoded values) and the
e4m3 one also to torch's own float32 -> float8_e4m3fn conversion; the scaling
rules to their closed forms (amax / 448 per token; OCP MX v1.0 shared exponent
floor(log2 amax) - 2 per 32-element block); the scatter to the slot mapping
(only the addressed rows change, in any slot order)."""
import math

import numpy as np
import pytest
import torch

import oracle


def nearest_code(v, values, codes):
    """Brute force: the code whose value is nearest to v; ties to the even code."""
    best = None
    for c, x in zip(codes, values):
        d = abs(x - v)
        if best is None or d < best[0] - 1e-300 or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return best[1]


def test_encode_e4m3_brute_force_and_torch():
    mags = [oracle.decode_e4m3(c) for c in range(0x7F)]           # 0 .. 448, codes 0x00 .. 0x7E
    codes = list(range(0x7F))
    g = torch.Generator().manual_seed(3)
    vals = torch.cat([torch.randn(3000, generator=g) * s for s in (1e-3, 0.05, 1.0, 40.0, 200.0)])
    # exact midpoints between neighbouring codes (ties) and the grid itself
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(len(mags) - 1)]
    vals = torch.cat([vals, torch.tensor(mags + mids, dtype=torch.float32),
                      -torch.tensor(mids, dtype=torch.float32)])
    vals = vals.to(torch.float32)
    ours = [oracle.encode_e4m3(float(v)) for v in vals]
    ref_torch = vals.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    for v, o, t in zip(vals.tolist(), ours, ref_torch):
        a = abs(v)
        want = nearest_code(a, mags, codes) | (0x80 if math.copysign(1.0, v) < 0 else 0)
        assert o == want, (v, o, want)
        if a < 464.0:                      # torch rounds up to its NaN code beyond this
            assert o == t, (v, o, t)
    # saturation (torch gives NaN above the rounding range; the scatter never feeds it such values)
    assert oracle.encode_e4m3(448.0) == 0x7E and oracle.encode_e4m3(1e6) == 0x7E
    assert oracle.encode_e4m3(-500.0) == 0xFE
    assert oracle.encode_e4m3(0.0) == 0x00 and oracle.encode_e4m3(-0.0) == 0x80


def test_encode_e2m1_brute_force_and_ties():
    mags = [oracle.decode_e2m1(c) for c in range(8)]
    assert mags == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    g = torch.Generator().manual_seed(4)
    vals = (torch.rand(4000, generator=g) * 8 - 4).tolist()
    vals += [(mags[i] + mags[i + 1]) / 2 for i in range(7)] + mags + [5.9, 6.1, 100.0]
    for v in vals:
        v = float(np.float32(v))
        want = nearest_code(abs(v), mags, list(range(8))) | (8 if math.copysign(1.0, v) < 0 else 0)
        assert oracle.encode_e2m1(v) == want, v
    # the ties explicitly: to the even code
    assert [oracle.encode_e2m1(x) for x in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 2, 2, 4, 4, 6, 6]


def make_cache(fmt, D, P, pages, vpad=0, spad=0):
    tok = D if fmt == 0 else D // 2
    stok = 4 if fmt == 0 else D // 32
    vps, sps = P * tok + vpad, P * stok + spad
    vals = np.full(pages * vps, 0xEE, np.uint8)
    scs = np.full(pages * sps, 0xEE, np.uint8)
    bt = np.zeros((1, 1), np.int32)
    return oracle.PagedBytes(vals, vps, tok, scs, sps, stok, bt, P, pages)


def test_fp8_scatter_closed_form():
    D, P, pages = 64, 32, 4
    g = torch.Generator().manual_seed(5)
    k = torch.randn((6, D), generator=g) * torch.tensor([1, 10, 1e-3, 0, 300, 1])[:, None]
    slots = [5, 32 * 3 + 31, -1, 64, 1, 126]
    c = make_cache(0, D, P, pages, vpad=16)
    oracle.quantize_scatter(k, slots, 0, c)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        p, r = divmod(s, P)
        row = c.values[p * c.vps + r * c.vts: p * c.vps + r * c.vts + D]
        sc = c.scales[p * c.sps + r * c.sts: p * c.sps + r * c.sts + 4].view(np.float32)[0]
        x = k[t].numpy().astype(np.float32)
        amax = np.float32(np.max(np.abs(x)))
        want_sc = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        assert sc == want_sc
        want = torch.from_numpy((x / want_sc).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
        assert np.array_equal(row, want.numpy()), t
        # the largest element lands on the top of the grid (+-448), dequantised back within half a step
        if amax > 0:
            deq = np.array([oracle.decode_e4m3(int(b)) for b in row]) * float(sc)
            assert np.max(np.abs(deq - x)) <= amax / 448 * 16 + 1e-30
    # untouched: the padding and every slot not addressed
    touched = set(s for s in slots if s >= 0)
    for s in range(pages * P):
        if s in touched:
            continue
        p, r = divmod(s, P)
        assert np.all(c.values[p * c.vps + r * c.vts: p * c.vps + r * c.vts + D] == 0xEE)
    for p in range(pages):
        assert np.all(c.values[p * c.vps + P * D: (p + 1) * c.vps] == 0xEE)


def test_mxfp4_scatter_closed_form():
    D, P, pages = 64, 32, 2
    g = torch.Generator().manual_seed(6)
    k = torch.randn((5, D), generator=g)
    k[1, :32] *= 1e-4          # a small block
    k[2, 32:] = 0.0            # an all-zero block
    k[3] *= 1e3
    kb = k.to(torch.bfloat16)
    slots = [0, 33, 63, 7, -5]
    c = make_cache(1, D, P, pages, vpad=32, spad=16)
    oracle.quantize_scatter(kb, slots, 1, c)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        p, r = divmod(s, P)
        row = c.values[p * c.vps + r * c.vts: p * c.vps + r * c.vts + D // 2]
        sc = c.scales[p * c.sps + r * c.sts: p * c.sps + r * c.sts + D // 32]
        x = kb[t].float().numpy()
        for blk in range(D // 32):
            xb = x[32 * blk: 32 * blk + 32]
            amax = float(np.max(np.abs(xb)))
            e = (math.frexp(amax)[1] - 1 - 2) if amax > 0 else -127
            e = max(-127, min(127, e))
            assert int(sc[blk]) == e + 127, (t, blk)
            for j in range(32):
                d = 32 * blk + j
                nib = (int(row[d // 2]) >> (4 * (d % 2))) & 0xF
                assert nib == oracle.encode_e2m1(float(np.float32(xb[j] * 2.0 ** -e))), (t, d)
            # the block's largest magnitude is within the e2m1 range after scaling: [4, 8) before saturation
            if amax > 0:
                assert 4.0 <= amax * 2.0 ** -e < 8.0


def test_scatter_order_invariance():
    """The slot order does not matter (each slot is written once)."""
    D, P, pages = 128, 64, 3
    g = torch.Generator().manual_seed(7)
    k = torch.randn((40, D), generator=g)
    slots = np.random.default_rng(0).permutation(pages * P)[:40]
    for fmt in (0, 1):
        a = make_cache(fmt, D, P, pages)
        b = make_cache(fmt, D, P, pages)
        oracle.quantize_scatter(k, slots, fmt, a)
        perm = np.random.default_rng(1).permutation(40)
        oracle.quantize_scatter(k[torch.from_numpy(perm)], slots[perm], fmt, b)
        assert np.array_equal(a.values, b.values) and np.array_equal(a.scales, b.scales)


def test_scatter_then_logits_round_trip():
    """Quantising exactly representable rows reproduces them: a row whose values
    are e4m3 codes times a power-of-two scale with amax 448*scale is stored as
    those codes and that scale."""
    D, P = 32, 32
    codes = torch.randint(0, 0x7E, (3, D), generator=torch.Generator().manual_seed(8)).to(torch.uint8)
    codes[:, 0] = 0x7E                                                  # amax element = 448
    vals = codes.view(torch.float8_e4m3fn).float() * 0.25
    c = make_cache(0, D, P, 1)
    oracle.quantize_scatter(vals, [0, 1, 2], 0, c)
    for t in range(3):
        assert np.array_equal(c.values[t * D:(t + 1) * D], codes[t].numpy())
        assert c.scales[4 * t: 4 * t + 4].view(np.float32)[0] == 0.25
