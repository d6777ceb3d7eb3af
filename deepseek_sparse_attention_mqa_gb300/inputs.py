"""Seeded synthetic inputs for the sparse-attention decode path.

This module only draws random numbers and lays bytes out in memory; it holds
none of the method's arithmetic (no decoding, no dot products, no masking, no
selection, no softmax).  Both the CUDA path and the CPU oracle consume what it
produces, so it is the one module they share.

Shapes and distributions follow the workloads of the pages' test matrices
("SM120 FP8 paged MQA page 32": page 32/64, heads 16..64, next_n 1..3 +
varlen, shuffled physical pages, padded page strides, empty history, partial
pages) and the five named workloads:

* ``tiny``       batch 2, next_n 1, H 4, D 32, page 64, lens {200, 317}, top-k 64,
                 MLA 4 heads over a bf16 latent (q/k 80, v 64)
* ``decode``     batch 64, next_n 1, H 64, D 128, page 64, lens U[4096, 32768],
                 2x oversized pool, top-k 2048
* ``spec_mxfp4`` batch 128, next_n 2, H 32, D 64, page 32, lens log-uniform in
                 [0, 65536] (+ forced edge lengths), MXFP4, padded strides, top-k 512
* ``prefill``    one causal sequence of 16384 tokens, H 64, D 128, page 64, top-k 2048
* ``full_step``  batch 64, next_n 1, H 4, D 32, page 64, lens U[8192, 131072], top-k 2048,
                 MLA 128 heads over an FP8 latent (q/k 576, v 512), scale 1/sqrt(192)
* ``full_step_h64``  the same with the decode indexer shape, H 64, D 128

Draw order (one ``torch.Generator`` seeded with ``seed``): context lengths,
physical page permutation, K values, K scales, q, weights, then the MLA latent
values, latent scales and MLA q.  Unused pool pages and stride padding hold
NaN codes (0x7F for e4m3 / e2m1 pairs, NaN for fp32 scales, 0xFF for ue8m0)
so that a stray read shows up against the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

FMT_FP8 = 0
FMT_MXFP4 = 1
FMT_BF16 = 2

NAN_BYTE = 0x7F


@dataclass
class Paged:
    """A paged cache as raw bytes.  ``values`` is [num_pages, val_page_stride]
    uint8; token t of page p starts at byte p*val_page_stride + t*val_token_stride.
    ``scales`` likewise (fp32 per token for FP8, ue8m0 per 32 elements for MXFP4,
    None for bf16)."""
    fmt: int
    head_dim: int
    page_kv: int
    num_pages: int
    values: torch.Tensor
    val_page_stride: int
    val_token_stride: int
    scales: Optional[torch.Tensor]
    sc_page_stride: int
    sc_token_stride: int


@dataclass
class Case:
    name: str
    batch: int
    next_n: int
    num_heads: int
    head_dim: int
    page_kv: int
    fmt: int
    topk: int
    width: int                      # logits row capacity (max visible entries)
    context_lens: torch.Tensor      # [batch] int32
    block_table: torch.Tensor       # [batch, max_pages] int32, -1 where unused
    kcache: Paged
    q: torch.Tensor                 # [R, H, D] e4m3 bytes, or [R, H, D/2] packed e2m1
    q_scales: Optional[torch.Tensor]  # [R, H, D/32] ue8m0 (MXFP4 only)
    weights: torch.Tensor           # [R, H] fp32
    # sparse MLA (optional)
    mla_heads: int = 0
    d_qk: int = 0
    d_v: int = 0
    softmax_scale: float = 0.0
    latent: Optional[Paged] = None
    q_mla: Optional[torch.Tensor] = None   # [R, Hq, d_qk] bf16
    meta: dict = field(default_factory=dict)
    ratio: int = 1                  # tokens per K-cache entry (compressed indexer cache)

    @property
    def rows(self) -> int:
        return self.batch * self.next_n


# ------------------------------------------------------------------ configs

CONFIGS = {
    "tiny": dict(batch=2, next_n=1, num_heads=4, head_dim=32, page_kv=64, fmt=FMT_FP8,
                 lens=("fixed", [200, 317]), pool_factor=1, w_div=math.sqrt(4), topk=64,
                 mla=dict(heads=4, d_qk=80, d_v=64, fmt=FMT_BF16, scale=1.0 / math.sqrt(80)),
                 seed=0),
    "decode": dict(batch=64, next_n=1, num_heads=64, head_dim=128, page_kv=64, fmt=FMT_FP8,
                   lens=("uniform", 4096, 32768), pool_factor=2, w_div=8.0, topk=2048,
                   width=32768, seed=1),
    "spec_mxfp4": dict(batch=128, next_n=2, num_heads=32, head_dim=64, page_kv=32,
                       fmt=FMT_MXFP4, lens=("loguniform", 65536), pool_factor=1,
                       w_div=math.sqrt(32), topk=512, width=65536, val_pad=1024, sc_pad=64,
                       seed=2),
    "prefill": dict(batch=1, next_n=16384, num_heads=64, head_dim=128, page_kv=64,
                    fmt=FMT_FP8, lens=("fixed", [16384]), pool_factor=1, w_div=8.0,
                    topk=2048, width=16384, seed=3),
    "full_step": dict(batch=64, next_n=1, num_heads=4, head_dim=32, page_kv=64, fmt=FMT_FP8,
                      lens=("uniform", 8192, 131072), pool_factor=1, w_div=math.sqrt(4),
                      topk=2048, width=131072,
                      mla=dict(heads=128, d_qk=576, d_v=512, fmt=FMT_FP8,
                               scale=1.0 / math.sqrt(192)),
                      seed=4),
    # the same step with the decode workload's indexer shape (64 heads x 128)
    "full_step_h64": dict(batch=64, next_n=1, num_heads=64, head_dim=128, page_kv=64, fmt=FMT_FP8,
                          lens=("uniform", 8192, 131072), pool_factor=1, w_div=8.0,
                          topk=2048, width=131072,
                          mla=dict(heads=128, d_qk=576, d_v=512, fmt=FMT_FP8,
                                   scale=1.0 / math.sqrt(192)),
                          seed=4),
}

# Lengths forced onto the first sequences of the log-uniform workload: empty
# history, one and two tokens, partial and exact pages, the maximum.
EDGE_LENS = [0, 1, 2, 31, 32, 33, 64, 65536]


def _lens(spec, batch, g):
    kind = spec[0]
    if kind == "fixed":
        return torch.tensor(spec[1], dtype=torch.int32)
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        top = spec[1]
        u = torch.rand((batch,), generator=g, dtype=torch.float64)
        L = torch.floor(torch.exp(u * math.log(top + 1))) - 1
        L = L.clamp(0, top).to(torch.int32)
        n = min(len(EDGE_LENS), batch)
        L[:n] = torch.tensor(EDGE_LENS[:n], dtype=torch.int32)
        return L
    raise ValueError(kind)


def _to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


# e2m1 magnitude grid in code order 0..7 and the decision boundaries between
# neighbours (ties go to the smaller magnitude; generator rounding only).
_E2M1_BOUNDS = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]


def mxfp4_quantize(x: torch.Tensor):
    """Quantise the last dim of ``x`` (a multiple of 32) to MXFP4 following the
    OCP MX v1.0 recipe: per 32-element block, shared exponent
    floor(log2(amax)) - 2 stored as ue8m0, elements divided by 2^exp and
    rounded onto the e2m1 grid with saturation at 6.  Returns (packed bytes
    [..., D/2] with the even element in the low nibble, ue8m0 [..., D/32])."""
    *lead, D = x.shape
    assert D % 32 == 0
    xb = x.to(torch.float32).reshape(*lead, D // 32, 32)
    amax = xb.abs().amax(dim=-1, keepdim=True)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax.clamp_min(1e-38))) - 2,
                    torch.full_like(amax, -127.0))
    e = e.clamp(-127, 127)
    scaled = xb / torch.exp2(e)
    mag = scaled.abs().clamp(max=6.0)
    bounds = torch.tensor(_E2M1_BOUNDS, dtype=torch.float32, device=x.device)
    code = torch.bucketize(mag.contiguous(), bounds, right=False).to(torch.uint8)
    sign = ((scaled < 0) & (code > 0)).to(torch.uint8) << 3
    nib = (code | sign).reshape(*lead, D)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).contiguous()
    sc = (e + 127).to(torch.int32).clamp(0, 254).to(torch.uint8).reshape(*lead, D // 32)
    return packed, sc


def _layout_pages(page_data: torch.Tensor, num_pages: int, page_stride: int, fill: int):
    """Place dense per-page bytes [num_pages, dense] into [num_pages, page_stride]
    with the tail of each page (stride padding) holding ``fill``."""
    dense = page_data.shape[1]
    out = torch.full((num_pages, page_stride), fill, dtype=torch.uint8, device=page_data.device)
    out[:, :dense] = page_data
    return out


def make_case(name: str, seed: Optional[int] = None, device="cpu", batch: Optional[int] = None,
              lens=None, with_mla: bool = True, **over) -> Case:
    """Build one workload.  ``batch``/``lens``/``over`` shrink or vary it for
    tests (e.g. fewer sequences, other page sizes); ``lens`` replaces the
    length draw with explicit context lengths."""
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    if seed is None:
        seed = cfg["seed"]
    if batch is not None:
        cfg["batch"] = batch
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    gc = torch.Generator()           # CPU stream for the small integer draws
    gc.manual_seed(int(seed))

    B, n, H, D, P = cfg["batch"], cfg["next_n"], cfg["num_heads"], cfg["head_dim"], cfg["page_kv"]
    fmt = cfg["fmt"]
    if lens is not None:
        L = torch.tensor(list(lens), dtype=torch.int32)
        B = L.numel()
    else:
        L = _lens(cfg["lens"], B, gc)
        B = L.numel()
    R = B * n
    # a compressed K cache (ratio > 1) holds one entry per `ratio` tokens
    ratio = int(cfg.get("ratio", 1))
    entries = [int(l) // ratio for l in L.tolist()]
    width = int(cfg.get("width", 0)) or (max(entries) if B else 0)
    width = max(width, max(entries) if B else 0)
    pages_per_seq = [(e + P - 1) // P for e in entries]
    used = sum(pages_per_seq)
    pool = max(1, used * int(cfg.get("pool_factor", 1)))
    max_pages = max(1, (width + P - 1) // P)

    perm = torch.randperm(pool, generator=gc)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, np_ in enumerate(pages_per_seq):
        bt[b, :np_] = perm[pos:pos + np_].to(torch.int32)
        pos += np_
    used_mask = torch.zeros(pool, dtype=torch.bool)
    used_mask[perm[:used]] = True
    used_mask = used_mask.to(dev)

    # ---- indexer K cache
    if fmt == FMT_FP8:
        tok_bytes = D
        vals = _to_e4m3_bytes(torch.randn((pool, P, D), generator=g, device=dev))
        vals[~used_mask] = NAN_BYTE
        val_pad = int(cfg.get("val_pad", 0))
        vstride = P * tok_bytes + val_pad
        values = _layout_pages(vals.reshape(pool, P * tok_bytes), pool, vstride, NAN_BYTE)
        sc = torch.rand((pool, P), generator=g, device=dev) * 1.5 + 0.5
        sc[~used_mask] = float("nan")
        sc_pad = int(cfg.get("sc_pad", 0))
        sstride = P * 4 + sc_pad
        scales = _layout_pages(sc.contiguous().view(torch.uint8).reshape(pool, P * 4), pool,
                               sstride, 0xFF)
        kc = Paged(FMT_FP8, D, P, pool, values, vstride, tok_bytes, scales, sstride, 4)
        q = _to_e4m3_bytes(torch.randn((R, H, D), generator=g, device=dev))
        q_scales = None
    elif fmt == FMT_MXFP4:
        tok_bytes = D // 2
        kx = torch.randn((pool, P, D), generator=g, device=dev)
        kp, ks = mxfp4_quantize(kx)
        kp[~used_mask] = NAN_BYTE
        ks[~used_mask] = 0xFF
        val_pad = int(cfg.get("val_pad", 0))
        vstride = P * tok_bytes + val_pad
        values = _layout_pages(kp.reshape(pool, P * tok_bytes), pool, vstride, NAN_BYTE)
        sc_pad = int(cfg.get("sc_pad", 0))
        sstride = P * (D // 32) + sc_pad
        scales = _layout_pages(ks.reshape(pool, P * (D // 32)), pool, sstride, 0xFF)
        kc = Paged(FMT_MXFP4, D, P, pool, values, vstride, tok_bytes, scales, sstride, D // 32)
        q, q_scales = mxfp4_quantize(torch.randn((R, H, D), generator=g, device=dev))
    else:
        raise ValueError("indexer format %d" % fmt)
    w = torch.randn((R, H), generator=g, device=dev) / float(cfg["w_div"])

    case = Case(name=name, batch=B, next_n=n, num_heads=H, head_dim=D, page_kv=P, fmt=fmt,
                topk=int(cfg["topk"]), width=width, context_lens=L.to(dev),
                block_table=bt.to(dev), kcache=kc, q=q.contiguous(),
                q_scales=None if q_scales is None else q_scales.contiguous(),
                weights=w.contiguous(), meta=dict(seed=int(seed), pool=pool, used_pages=used), ratio=ratio)

    mla = cfg.get("mla")
    if with_mla and mla:
        Hq, dqk, dv = mla["heads"], mla["d_qk"], mla["d_v"]
        if mla["fmt"] == FMT_FP8:
            lv = _to_e4m3_bytes(torch.randn((pool, P, dqk), generator=g, device=dev))
            lv[~used_mask] = NAN_BYTE
            lvals = lv.reshape(pool, P * dqk).contiguous()
            ls = torch.rand((pool, P), generator=g, device=dev) * 1.5 + 0.5
            ls[~used_mask] = float("nan")
            lscales = ls.contiguous().view(torch.uint8).reshape(pool, P * 4)
            lat = Paged(FMT_FP8, dqk, P, pool, lvals, P * dqk, dqk, lscales, P * 4, 4)
        else:
            lv = torch.randn((pool, P, dqk), generator=g, device=dev).to(torch.bfloat16)
            lvals = lv.view(torch.uint8).reshape(pool, P * dqk * 2).contiguous()
            lat = Paged(FMT_BF16, dqk, P, pool, lvals, P * dqk * 2, dqk * 2, None, 0, 0)
        qm = torch.randn((R, Hq, dqk), generator=g, device=dev).to(torch.bfloat16)
        case.mla_heads, case.d_qk, case.d_v = Hq, dqk, dv
        case.softmax_scale = float(mla["scale"])
        case.latent = lat
        case.q_mla = qm.contiguous()
    return case


def to_device(case: Case, device) -> Case:
    """Copy every tensor of a case to ``device`` (same bytes)."""
    import copy
    c = copy.copy(case)
    dev = torch.device(device)
    for f in ("context_lens", "block_table", "q", "q_scales", "weights", "q_mla"):
        t = getattr(c, f)
        if t is not None:
            setattr(c, f, t.to(dev))
    for f in ("kcache", "latent"):
        p = getattr(c, f)
        if p is not None:
            p2 = copy.copy(p)
            p2.values = p.values.to(dev)
            p2.scales = None if p.scales is None else p.scales.to(dev)
            setattr(c, f, p2)
    return c


@dataclass
class SwaCase:
    """Sparse MLA over two latent caches: a compressed ("sparse") cache whose
    entries are selected per row by ``idx`` (the first ``topk_lens[r]`` of
    them), and a sliding-window cache of the sequence's tokens.  Rows of
    sequence b are [cum_q[b], cum_q[b + 1]); ``seq_lens`` counts each sequence's
    tokens including its new ones."""
    batch: int
    rows: int
    heads: int
    d_qk: int
    d_v: int
    fmt: int
    softmax_scale: float
    k: int
    window: int
    seq_lens: torch.Tensor          # [batch] int32
    cum_q: torch.Tensor             # [batch + 1] int32
    sparse: Paged
    sparse_bt: torch.Tensor         # [batch, max_pages] int32
    swa: Paged
    swa_bt: torch.Tensor            # [batch, max_pages] int32
    idx: torch.Tensor               # [rows, k] int32, -1 padding
    topk_lens: torch.Tensor         # [rows] int32
    q: torch.Tensor                 # [rows, heads, d_qk] bf16


def _latent_pool(pages, P, D, fmt, g, dev):
    if fmt == FMT_FP8:
        v = _to_e4m3_bytes(torch.randn((pages, P, D), generator=g, device=dev)).reshape(pages, P * D).contiguous()
        s = (torch.rand((pages, P), generator=g, device=dev) * 1.5 + 0.5).contiguous()
        return Paged(FMT_FP8, D, P, pages, v, P * D, D, s.view(torch.uint8).reshape(pages, P * 4), P * 4, 4)
    v = torch.randn((pages, P, D), generator=g, device=dev).to(torch.bfloat16)
    return Paged(FMT_BF16, D, P, pages, v.view(torch.uint8).reshape(pages, P * D * 2).contiguous(), P * D * 2,
                 D * 2, None, 0, 0)


def _pages_for(lengths, P, gc):
    """Block table [batch, max_pages] over a shuffled pool covering `lengths`."""
    per = [(int(l) + P - 1) // P for l in lengths]
    pool = max(1, sum(per))
    perm = torch.randperm(pool, generator=gc)
    bt = torch.full((len(per), max(1, max(per) if per else 1)), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(per):
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    return bt, pool


def make_swa_case(seed=0, device="cpu", seq_lens=(300, 1000, 70), q_lens=(1, 3, 2), heads=16, d_qk=576,
                  d_v=512, fmt=FMT_FP8, page_kv=64, swa_page_kv=64, k=128, window=128, ratio=4,
                  scale=None) -> SwaCase:
    """Random two-cache sparse MLA workload: each sequence's sparse cache holds
    seq_len // ratio + 1 entries; each row selects k of them at random (a few
    slots -1) and keeps a random leading count topk_lens[r] in [0, k]."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    gc = torch.Generator()
    gc.manual_seed(int(seed))
    L = torch.tensor(list(seq_lens), dtype=torch.int32)
    ql = list(q_lens)
    B = len(ql)
    cum = torch.zeros(B + 1, dtype=torch.int32)
    cum[1:] = torch.cumsum(torch.tensor(ql, dtype=torch.int32), 0)
    R = int(cum[-1])
    n_sparse = [int(l) // ratio + 1 for l in L.tolist()]
    sbt, spool = _pages_for(n_sparse, page_kv, gc)
    wbt, wpool = _pages_for(L.tolist(), swa_page_kv, gc)
    idx = torch.full((R, k), -1, dtype=torch.int32)
    tl = torch.zeros(R, dtype=torch.int32)
    for b in range(B):
        for r in range(int(cum[b]), int(cum[b + 1])):
            take = min(k, n_sparse[b])
            sel = torch.randperm(n_sparse[b], generator=gc)[:take].to(torch.int32)
            idx[r, :take] = sel
            if take > 4:
                idx[r, torch.randint(0, take, (2,), generator=gc)] = -1
            tl[r] = int(torch.randint(0, k + 1, (1,), generator=gc))
    sparse = _latent_pool(spool, page_kv, d_qk, fmt, g, dev)
    swa = _latent_pool(wpool, swa_page_kv, d_qk, fmt, g, dev)
    q = torch.randn((R, heads, d_qk), generator=g, device=dev).to(torch.bfloat16).contiguous()
    return SwaCase(batch=B, rows=R, heads=heads, d_qk=d_qk, d_v=d_v, fmt=fmt,
                   softmax_scale=float(scale if scale is not None else 1.0 / math.sqrt(192)), k=k, window=window,
                   seq_lens=L.to(dev), cum_q=cum.to(dev), sparse=sparse, sparse_bt=sbt.to(dev), swa=swa,
                   swa_bt=wbt.to(dev), idx=idx.to(dev), topk_lens=tl.to(dev), q=q)
