"""One sparse-attention step over caller-owned device buffers.

A step is: build the indexer schedule on the device, score the paged
lightning-indexer logits, select the per-row top-k, and (when the workload has
an MLA stage) run sparse MLA decode over the selected latent tokens.  Prefill
rows are processed in chunks so that the fp32 logits buffer stays within a
byte budget ("feat(deepseek_v4): Add fp4 indexer for dsv4", prefill notes:
logits width = the actual longest visible length, Q-row budget chunking, one
schedule per chunk).  Every step of the computation runs in libdsa; this
module only allocates buffers once and issues the C-ABI calls in order, so the
whole step can be captured in one CUDA graph.
"""
from __future__ import annotations

import torch

from . import _abi
from .inputs import Case

LOGITS_BUDGET_BYTES = 512 * 1024 * 1024   # 512 MiB


class StepInputs:
    """The query-side inputs of a step (indexer q and its block scales, head
    weights, context lengths, block table, and the MLA q when present) packed
    into one device arena and one pinned host arena of the same layout, so that
    a serving loop moves a step's inputs with ONE host-to-device copy instead of
    one per tensor (each copy costs a few microseconds of issue latency on its
    own).  ``case()`` returns the workload rebound to the device views; write a
    step's inputs into ``host[name]`` and call ``copy_in()``."""

    NAMES = ("q", "q_scales", "weights", "context_lens", "block_table", "q_mla")

    def __init__(self, case: Case, with_mla: bool = True):
        import dataclasses
        dev = case.q.device
        names = self.NAMES if with_mla else self.NAMES[:-1]
        tensors = {n: getattr(case, n) for n in names if getattr(case, n) is not None}
        offs, total = {}, 0
        for n, t in tensors.items():
            offs[n] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = total
        self.device_arena = torch.empty((max(total, 256),), dtype=torch.uint8, device=dev)
        self.host_arena = torch.empty((max(total, 256),), dtype=torch.uint8).pin_memory()

        def view(arena, n, t):
            nb = t.numel() * t.element_size()
            return arena[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)

        self.device = {n: view(self.device_arena, n, t) for n, t in tensors.items()}
        self.host = {n: view(self.host_arena, n, t) for n, t in tensors.items()}
        for n, t in tensors.items():
            self.host[n].copy_(t.cpu())
            self.device[n].copy_(t)
        self._case = dataclasses.replace(case, **self.device)

    def case(self) -> Case:
        return self._case

    def copy_in(self, stream=None):
        """Enqueue the one host-to-device copy of every input on `stream`."""
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            self.device_arena.copy_(self.host_arena, non_blocking=True)


class SparseAttentionStep:
    def __init__(self, case: Case, with_mla: bool = True, budget_bytes: int = LOGITS_BUDGET_BYTES,
                 rows_per_chunk: int | None = None, inline_schedule: bool | None = None,
                 fused: bool = False):
        dev = case.q.device
        assert dev.type == "cuda", "SparseAttentionStep needs the case on a CUDA device"
        self.case = case
        c = case
        self.rows = c.rows
        self.width = int(c.width)
        if rows_per_chunk is None:
            rows_per_chunk = max(1, min(self.rows, budget_bytes // (4 * max(1, self.width))))
        self.rows_per_chunk = int(rows_per_chunk)
        self.chunks = [(rb, min(self.rows, rb + self.rows_per_chunk))
                       for rb in range(0, self.rows, self.rows_per_chunk)] or [(0, 0)]
        kc = c.kcache
        self.ratio = int(getattr(c, "ratio", 1))
        self.kcache = _abi.make_cache(kc.fmt, kc.head_dim, kc.page_kv, kc.num_pages, kc.values,
                                      kc.val_page_stride, kc.val_token_stride, kc.scales,
                                      kc.sc_page_stride, kc.sc_token_stride, c.block_table,
                                      compress_ratio=self.ratio)
        # a chunk of at most INLINE_UNITS units needs no schedule launch: the logits
        # kernel builds its units itself (inline_schedule=False forces the buffer)
        self.inline = {(rb, re): (inline_schedule is not False and
                                  _abi.units_of(c.batch, c.next_n, c.num_heads, rb, re) <= _abi.INLINE_UNITS)
                       for rb, re in self.chunks}
        sb = max(_abi.schedule_bytes(c.batch, c.next_n, c.num_heads, rb, re) for rb, re in self.chunks)
        self.sched = torch.empty((sb + 15) // 16 * 4, dtype=torch.int32, device=dev)
        self.logits = torch.empty((self.rows_per_chunk, max(1, self.width)), dtype=torch.float32,
                                  device=dev)
        self.idx = torch.empty((self.rows, c.topk), dtype=torch.int32, device=dev)
        self.count = torch.empty((self.rows,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        tw = _abi.topk_workspace_bytes(self.rows_per_chunk, self.width, c.topk)
        self.topk_ws = torch.empty((max(tw, 16),), dtype=torch.uint8, device=dev)
        # fused score + top-k: one launch per chunk; its per-unit counters start at
        # zero and every call leaves them at zero
        self.fused = bool(fused)
        if self.fused:
            fw = max(_abi.score_topk_workspace_bytes(c.batch, c.next_n, c.num_heads, rb, re)
                     for rb, re in self.chunks)
            self.fused_ws = torch.zeros(((fw + 15) // 16 * 4,), dtype=torch.int32, device=dev)
        self.with_mla = bool(with_mla and c.latent is not None)
        if self.with_mla:
            lat = c.latent
            self.latent = _abi.make_cache(lat.fmt, lat.head_dim, lat.page_kv, lat.num_pages,
                                          lat.values, lat.val_page_stride, lat.val_token_stride,
                                          lat.scales, lat.sc_page_stride, lat.sc_token_stride,
                                          c.block_table)
            self.out = torch.empty((self.rows, c.mla_heads, c.d_v), dtype=torch.bfloat16, device=dev)
            self.lse = torch.empty((self.rows, c.mla_heads), dtype=torch.float32, device=dev)
            mw = _abi.mla_workspace_bytes(self.rows, c.mla_heads, c.d_qk, c.d_v, c.topk)
            self.mla_ws = torch.empty((max(mw, 16),), dtype=torch.uint8, device=dev)

    # ------------------------------------------------------------------ stages
    def indexer_chunk(self, rb: int, re: int, stream=None):
        c = self.case
        inline = self.inline.get((rb, re), False)
        if not inline:
            _abi.build_schedule(c.context_lens, c.batch, c.next_n, c.num_heads, rb, re, self.sched,
                                self.status, stream, compress_ratio=self.ratio)
        _abi.mqa_logits(c.q, c.q_scales, c.fmt, c.weights, c.num_heads, self.kcache,
                        c.context_lens, c.batch, c.next_n, rb, re, None if inline else self.sched,
                        self.logits, self.width, self.status, stream)

    def score_topk_chunk(self, rb: int, re: int, stream=None):
        """Logits and top-k of rows [rb, re) in one fused launch (plus the
        schedule launch for chunks of more than INLINE_UNITS units)."""
        c = self.case
        inline = self.inline.get((rb, re), False)
        if not inline:
            _abi.build_schedule(c.context_lens, c.batch, c.next_n, c.num_heads, rb, re, self.sched,
                                self.status, stream, compress_ratio=self.ratio)
        _abi.score_topk(c.q, c.q_scales, c.fmt, c.weights, c.num_heads, self.kcache, c.context_lens,
                        c.batch, c.next_n, rb, re, None if inline else self.sched, self.logits,
                        self.width, c.topk, self.idx[rb:re], self.count[rb:re], self.fused_ws,
                        self.status, stream)

    def topk_chunk(self, rb: int, re: int, stream=None):
        c = self.case
        _abi.topk(self.logits, self.width, c.context_lens, c.batch, c.next_n, rb, re, c.topk,
                  self.idx[rb:re], self.count[rb:re], self.topk_ws, self.status, stream,
                  compress_ratio=self.ratio)

    def mla(self, stream=None):
        c = self.case
        _abi.sparse_mla(c.q_mla, c.softmax_scale, self.latent, self.idx, c.topk, self.out,
                        self.lse, c.d_v, None, c.next_n, self.mla_ws, self.status, stream)

    def run(self, stream=None):
        for rb, re in self.chunks:
            if re > rb:
                if self.fused:
                    self.score_topk_chunk(rb, re, stream)
                else:
                    self.indexer_chunk(rb, re, stream)
                    self.topk_chunk(rb, re, stream)
        if self.with_mla:
            self.mla(stream)

    def launches_per_step(self) -> int:
        per = 1 if self.fused else 2
        n = sum(per + (0 if self.inline.get((rb, re), False) else 1) for rb, re in self.chunks if re > rb)
        return n + (1 if self.with_mla else 0)

    def device_status(self) -> int:
        return _abi.device_status(self.status)


class HostStepPipeline:
    """Steps fed from pinned host memory with their copies overlapped, the way a
    serving loop runs: two slots, each with its own input arena
    (``StepInputs``), step buffers and pinned result buffer, and three streams.
    The inputs of step i are copied in on the input stream once step i - 2 (the
    slot's previous user) has finished computing; step i runs on the compute
    stream once its inputs are in; its top-k indices go back to the host on the
    output stream once it has run.  So the copies of step i + 1 and step i - 1
    overlap the computation of step i.

    ``submit()`` enqueues one step and returns its slot; ``results(slot)`` waits
    for that slot's indices and returns the pinned host tensor (valid until the
    slot is submitted again).  Write a step's inputs into ``inputs[slot].host``
    before submitting it to that slot.  With ``graphs`` (the default) each
    slot's computation is captured once in a CUDA graph and replayed, so a
    submission costs the host two copies, four event operations and one replay
    instead of one library call per kernel.  With ``overlap_steps`` the two
    slots compute on streams of their own, so step i + 1 may start while step i
    finishes: for independent batches (two decode steps of the same sequences
    depend on each other and must not overlap)."""

    def __init__(self, case: Case, with_mla: bool = False, fused: bool = False, graphs: bool = True,
                 overlap_steps: bool = False):
        self.inputs = [StepInputs(case, with_mla=with_mla) for _ in range(2)]
        self.steps = [SparseAttentionStep(ins.case(), with_mla=with_mla, fused=fused) for ins in self.inputs]
        self.idx_host = [torch.empty(st.idx.shape, dtype=torch.int32).pin_memory() for st in self.steps]
        self.h2d_stream = torch.cuda.Stream()
        self.compute_stream = torch.cuda.Stream()
        # with overlap_steps each slot computes on its own stream, so step i + 1 may
        # start while step i finishes (the slots share no buffers)
        self.compute_streams = ([self.compute_stream, torch.cuda.Stream()] if overlap_steps
                                else [self.compute_stream, self.compute_stream])
        self.d2h_stream = torch.cuda.Stream()
        self._in_ready = [torch.cuda.Event() for _ in range(2)]
        self._computed = [torch.cuda.Event() for _ in range(2)]
        self._out_ready = [torch.cuda.Event() for _ in range(2)]
        self._used = [False, False]
        self._next = 0
        # the arenas were filled on the current stream at construction
        for s in (self.h2d_stream, self.d2h_stream, *self.compute_streams):
            s.wait_stream(torch.cuda.current_stream())
        self.graphs = None
        if graphs:
            with torch.cuda.stream(self.compute_stream):
                for st in self.steps:                   # warm-up outside the capture
                    st.run(self.compute_stream)
            self.compute_stream.synchronize()
            self.graphs = []
            for st in self.steps:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.compute_stream):
                    st.run(self.compute_stream)
                self.graphs.append(g)
            self.compute_stream.synchronize()

    @property
    def h2d_bytes(self) -> int:
        return self.inputs[0].nbytes

    @property
    def d2h_bytes(self) -> int:
        return self.idx_host[0].numel() * self.idx_host[0].element_size()

    def submit(self) -> int:
        s = self._next
        self._next ^= 1
        if self._used[s]:
            # the slot's device inputs are step i - 2's until it has computed
            self.h2d_stream.wait_event(self._computed[s])
        self.inputs[s].copy_in(self.h2d_stream)
        self._in_ready[s].record(self.h2d_stream)
        cs = self.compute_streams[s]
        cs.wait_event(self._in_ready[s])
        if self.graphs is not None:
            with torch.cuda.stream(cs):
                self.graphs[s].replay()
        else:
            self.steps[s].run(cs)
        self._computed[s].record(cs)
        self.d2h_stream.wait_event(self._computed[s])
        with torch.cuda.stream(self.d2h_stream):
            self.idx_host[s].copy_(self.steps[s].idx, non_blocking=True)
        self._out_ready[s].record(self.d2h_stream)
        self._used[s] = True
        return s

    def results(self, slot: int) -> torch.Tensor:
        self._out_ready[slot].synchronize()
        return self.idx_host[slot]

    def synchronize(self) -> None:
        for s in (self.h2d_stream, self.d2h_stream, *self.compute_streams):
            s.synchronize()
