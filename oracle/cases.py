"""Adapters from the seeded workloads (``deepseek_sparse_attention_mqa_gb300.inputs``)
to the oracle's inputs.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests, the smoke
check and the benchmark's CPU-baseline and reference legs use it; the CUDA
path never does.  Nothing here computes any part of the method: it copies the
bytes of a paged cache (optionally only some sequences' pages, renumbered) and
asks the oracle for a row's visible length.
"""
from __future__ import annotations

import torch

from . import PagedBytes, visible as _visible


def oracle_cache(paged, block_table, seqs=None):
    """(PagedBytes, seqs) from a (possibly device-resident) inputs.Paged.  With
    ``seqs`` only those sequences' pages are copied, renumbered in order, and
    row j of the returned block table is sequence seqs[j]; this keeps
    full-size workloads cheap to check on sampled rows."""
    bt = block_table.detach().cpu()
    if seqs is None:
        vals = paged.values.detach().cpu()
        scs = None if paged.scales is None else paged.scales.detach().cpu()
        return PagedBytes(vals, paged.val_page_stride, paged.val_token_stride, scs,
                          paged.sc_page_stride, paged.sc_token_stride, bt, paged.page_kv,
                          paged.num_pages), list(range(bt.shape[0]))
    seqs = list(seqs)
    phys = []
    new_bt = torch.full((len(seqs), bt.shape[1]), -1, dtype=torch.int32)
    for j, b in enumerate(seqs):
        row = bt[b]
        for lp in range(row.shape[0]):
            p = int(row[lp])
            if p < 0:
                continue
            new_bt[j, lp] = len(phys)
            phys.append(p)
    idx = torch.tensor(phys if phys else [0], dtype=torch.long, device=paged.values.device)
    vals = paged.values.index_select(0, idx).cpu()
    scs = None if paged.scales is None else paged.scales.index_select(0, idx).cpu()
    return PagedBytes(vals, paged.val_page_stride, paged.val_token_stride, scs,
                      paged.sc_page_stride, paged.sc_token_stride, new_bt, paged.page_kv,
                      max(1, len(phys))), seqs


def visible(case, r):
    """Visible entries of absolute row r of a workload (the oracle's window rule,
    over the workload's compression ratio)."""
    b, i = divmod(r, case.next_n)
    return _visible(int(case.context_lens[b]), case.next_n, i, getattr(case, "ratio", 1))
