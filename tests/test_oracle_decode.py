"""Pins for the oracle's format decoders and visibility windows (CPU only).

Each decoder is checked against something other than itself: torch's own
float8 / bfloat16 conversions for every code, or (e2m1, which torch cannot
convert) the OCP MX value set plus a round trip through an independent
quantiser with its error bound.
"""
import math

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_mqa_gb300 import inputs


def test_e4m3_all_codes_match_torch(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode_e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_ue8m0_all_codes_match_torch(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.decode_ue8m0(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_bf16_codes_match_torch(oracle):
    g = torch.Generator().manual_seed(7)
    bits = torch.randint(0, 65536, (4096,), generator=g, dtype=torch.int32)
    bits = torch.cat([bits, torch.tensor([0, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x7F7F])])
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(int(b)) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e2m1_value_set_and_symmetry(oracle):
    # OCP MX v1.0: e2m1 magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}, codes 0..7
    # increasing, bit 3 the sign.
    mags = [oracle.decode_e2m1(c) for c in range(8)]
    assert sorted(set(mags)) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert all(a < b for a, b in zip(mags, mags[1:]))
    for c in range(1, 8):
        assert oracle.decode_e2m1(c | 8) == -mags[c]
    assert oracle.decode_e2m1(8) == 0.0


def test_mxfp4_round_trip_error_bound(oracle):
    """Decode(quantise(x)) is within half a grid step (x 2^e) of x for values in
    range: the quantiser (bucketing on grid midpoints) and the oracle's decoder
    (bit fields) are written independently, so a wrong bias, nibble order or
    scale would break the bound."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn((16, 64), generator=g)
    packed, sc = inputs.mxfp4_quantize(x)
    pk = packed.numpy()
    scn = sc.numpy()
    for r in range(x.shape[0]):
        for d in range(64):
            byte = int(pk[r, d // 2])
            nib = byte & 0xF if d % 2 == 0 else byte >> 4
            s = oracle.decode_ue8m0(int(scn[r, d // 32]))
            v = oracle.decode_e2m1(nib) * s
            xv = float(x[r, d])
            # grid spacing at |x|/s is at most 2 (between 4 and 6); clamp at 6*s
            step = 0.5 if abs(xv) / s < 2 else (1.0 if abs(xv) / s < 4 else 2.0)
            bound = 0.5 * step * s + max(0.0, abs(xv) - 6 * s)
            assert abs(v - xv) <= bound + 1e-12, (r, d, xv, v, s)
            assert math.copysign(1.0, v) == math.copysign(1.0, xv) or v == 0.0


@pytest.mark.parametrize("L,n,expect", [
    (5, 3, [3, 4, 5]),        # speculative rows see one more token each
    (1, 3, [0, 0, 1]),        # short history: clamp at 0
    (0, 3, [0, 0, 0]),        # empty history
    (7, 1, [7]),              # plain decode
    (4, 4, [1, 2, 3, 4]),     # causal prefill
    (2, 2, [1, 2]),
])
def test_visible_windows_hand_enumerated(oracle, L, n, expect):
    assert [oracle.visible(L, n, i) for i in range(n)] == expect
