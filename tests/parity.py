"""Comparison rules shared by the GPU parity tests (GPU result vs fp64 oracle).

Tolerances (the method's statement of the bar):
  logits  max|d| <= 1e-3 * max|logit| over the visible entries of the workload;
  top-k   identical index sets wherever the oracle's k-th and (k+1)-th logits
          differ by more than that tolerance, compared by value otherwise;
  MLA     bf16 output max-abs error <= 1e-2 beyond the output's own bf16
          rounding (half an ulp), LSE max-abs error <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

LOGIT_RTOL = 1e-3
MLA_OUT_ATOL = 1e-2
MLA_LSE_ATOL = 1e-3


# the workload -> oracle adapters live beside the oracle (the benchmark's CPU
# legs use them too); re-exported here for the tests
from oracle.cases import oracle_cache, visible  # noqa: E402,F401


def check_logits(gpu_rows, ref_rows, vis, scale=None, what="logits"):
    """gpu_rows / ref_rows: lists of 1-D arrays (row r's first vis[r] entries
    are compared).  ``scale`` = max|logit| of the workload (default: of these rows)."""
    if scale is None:
        scale = max([float(np.max(np.abs(r[:v]))) for r, v in zip(ref_rows, vis) if v > 0] + [0.0])
    tol = LOGIT_RTOL * scale
    worst = 0.0
    for j, (g, o, v) in enumerate(zip(gpu_rows, ref_rows, vis)):
        if v == 0:
            continue
        g = np.asarray(g[:v], np.float64)
        o = np.asarray(o[:v], np.float64)
        assert np.all(np.isfinite(g)), "%s row %d: non-finite GPU logits" % (what, j)
        d = float(np.max(np.abs(g - o)))
        worst = max(worst, d)
        assert d <= tol, "%s row %d: max|d| %.3e > tol %.3e (scale %.3e)" % (what, j, d, tol, scale)
    return worst, tol


def check_topk_same_input(gpu_idx, ref_idx, vis, k):
    """Top-k of the SAME logits on both sides: the selected sets must be equal
    (index work, bit-exact); ties resolve to the lower position on both sides."""
    for j, v in enumerate(vis):
        take = min(k, v)
        g = np.asarray(gpu_idx[j])
        o = np.asarray(ref_idx[j])
        assert np.all(g[take:] == -1), "row %d: padding" % j
        assert sorted(g[:take].tolist()) == sorted(o[:take].tolist()), "row %d: index set" % j


def check_topk_tolerant(gpu_idx, ref_logits, vis, k, scale):
    """Top-k of the GPU logits vs the oracle logits: exact set where the oracle's
    k-th / (k+1)-th gap exceeds the tolerance, value rule otherwise."""
    tol = LOGIT_RTOL * scale
    exact_rows = 0
    for j, v in enumerate(vis):
        take = min(k, v)
        g = np.asarray(gpu_idx[j])
        assert np.all(g[take:] == -1), "row %d: padding" % j
        sel = g[:take]
        assert len(set(sel.tolist())) == take, "row %d: duplicate indices" % j
        assert np.all((sel >= 0) & (sel < v)), "row %d: index outside [0, vis)" % j
        if v <= k:
            continue
        o = np.asarray(ref_logits[j][:v], np.float64)
        order = np.argsort(-o, kind="stable")
        vk, vk1 = o[order[k - 1]], o[order[k]]
        if vk - vk1 > tol:
            assert set(sel.tolist()) == set(order[:k].tolist()), "row %d: set differs (gap %.3e)" % (j, vk - vk1)
            exact_rows += 1
        else:
            assert np.all(o[sel] >= vk - tol), "row %d: selected value below k-th - tol" % j
            must = np.nonzero(o > vk + tol)[0]
            assert set(must.tolist()) <= set(sel.tolist()), "row %d: missed a clearly larger logit" % j
    return exact_rows


def bf16_half_ulp(x):
    """Half a bf16 ulp at |x|: the rounding error of storing x in bf16."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), np.finfo(np.float64).tiny)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - 7)


def check_mla(out_gpu, lse_gpu, out_ref, lse_ref):
    """The output is bf16: its own rounding (half an ulp, up to 0.0156 at |x|
    ~ 8) is not kernel error, so the 1e-2 bound applies to the error beyond it:
    |gpu - oracle| <= 1e-2 + ulp_bf16(oracle)/2 elementwise."""
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    l = lse_gpu.detach().cpu().numpy().astype(np.float64)
    excess = np.abs(o - out_ref) - bf16_half_ulp(out_ref)
    eo = float(np.max(excess)) if o.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin), "LSE finiteness differs"
    assert np.all(l[~fin] == lse_ref[~fin])
    el = float(np.max(np.abs(l[fin] - lse_ref[fin]))) if fin.any() else 0.0
    assert eo <= MLA_OUT_ATOL, "MLA out error beyond bf16 rounding %.3e" % eo
    assert el <= MLA_LSE_ATOL, "MLA lse max-abs error %.3e" % el
    return eo, el
