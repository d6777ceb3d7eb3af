#!/usr/bin/env python3
"""Benchmark of the sparse-attention decode hot path on GB300.

Default workload (the decode indexer + top-k configuration): batch 64, next_n 1,
64 indexer heads, head_dim 128, page 64, context lengths U[4096, 32768] in a 2x
oversized shuffled FP8 pool, top-k 2048.  One step = device schedule build +
paged MQA logits + top-k (2 libdsa launches; the fused single-launch
indexer_score_topk is timed beside it, --fused makes it the headline).  Reported:

* value        K-tokens scored/s (sum of visible lengths / step time / 1e3),
               inputs resident in HBM, L2 flushed between steps, CUDA events;
* e2e          the same metric through the public step API with the step's
               query-side inputs (q, weights, context lengths, block table)
               copied from pinned host memory and the top-k indices copied back
               inside the timed region (the K cache is device-resident state);
* roofline     the logits kernel: algorithmic bytes per launch / its event time
               vs the measured HBM copy bandwidth;
* spec_mxfp4, prefill  the speculative/varlen MXFP4 and the causal prefill
               indexer configurations timed the same way (their own value,
               kernel times and roofline: HBM for MXFP4, FP8 tensor for prefill);
* kv_scatter   the K-cache quantise/scatter of a prefill's and a decode step's
               new tokens into FP8 and MXFP4 paged caches, with its HBM roofline;
* full_step    the whole graph-captured step of the full decode workload
               (indexer + top-k + sparse MLA, 128 heads 576/512) in us/step,
               with each stage also timed alone and the sparse MLA's tensor
               roofline; full_step_indexer_h64 is the same step with the decode
               indexer shape (64 heads x 128) in place of 4 heads x 32;
* cpu_baseline the fp64 oracle on the host cores over a bounded sample.

``--impl reference`` times the oracle itself (the only reference available
for this path) on the same workload and metric.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "indexer K-tokens scored/s & HBM GB/s (%roofline); sparse-attn decode µs/step"
UNIT = "K-tokens/s"
WORKLOAD = ("decode indexer + top-k: batch 64, next_n 1, 64 heads, head_dim 128, page 64, "
            "FP8 e4m3 K cache with fp32 token scale, lens U[4096,32768], 2x shuffled pool, top-k 2048")
WORKLOADS = {
    "decode": WORKLOAD,
    "spec_mxfp4": ("speculative/varlen indexer + top-k: batch 128, next_n 2, 32 heads, head_dim 64, "
                   "page 32, MXFP4 K cache and q in a padded-stride layout, lens log-uniform in "
                   "[0, 65536] with empty/partial-page edge lengths, top-k 512"),
    "prefill": ("prefill indexer + top-k: one causal sequence of 16384 tokens, 64 heads, head_dim 128, "
                "page 64, FP8 e4m3, logits width 16384, two 8192-row chunks (512 MiB budget), top-k 2048"),
}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.01)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_begin, t_end):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if t < t_begin - 0.15 or t > t_end + 0.15:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def scored_pairs(case):
    L = case.context_lens.cpu().tolist()
    n = case.next_n
    from deepseek_sparse_attention_mqa_gb300 import inputs as _  # noqa: F401
    tot = 0
    for b, l in enumerate(L):
        for i in range(n):
            v = l - n + i + 1
            tot += max(0, min(v, l))
    return tot


def logits_algorithmic_bytes(case):
    """Bytes the logits kernel must move: each sequence's visible K rows (values
    + scales) once, q (+ q scales) and weights once, the visible logits written once."""
    from deepseek_sparse_attention_mqa_gb300 import inputs
    D, H = case.head_dim, case.num_heads
    L = case.context_lens.cpu().tolist()
    if case.fmt == inputs.FMT_FP8:
        tok, qrow = D + 4, D
    else:
        tok, qrow = D // 2 + D // 32, D // 2 + D // 32
    kv = sum(l * tok for l in L)
    q = case.rows * H * qrow
    w = case.rows * H * 4
    out = scored_pairs(case) * 4
    bt = sum(-(-l // case.page_kv) for l in L) * 4 + len(L) * 4
    return kv + q + w + out + bt


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values of `x` (the job takes as long as its
    slowest replica); the value itself on one rank."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(pairs_per_replica: float, world: int, ms_per_step: float) -> float:
    """K-tokens scored per second over all replicas, each scoring the same
    workload in `ms_per_step` (the max over ranks)."""
    return pairs_per_replica * world / (ms_per_step * 1e-3) / 1e3


class L2Flush:
    """Evicts L2 (129 MB) between timed steps by READING a 384 MiB buffer (a
    reduction into one preallocated word): no dirty lines are left behind to be
    written back inside the next timed kernel.  At ~60 us of GPU time per flush
    it also keeps the GPU queue ahead of the host, so events time kernels, not
    host launch gaps."""

    BYTES = 384 * 2 ** 20

    def __init__(self, dev):
        self.buf = torch.ones(self.BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self, step=0):
        torch.sum(self.buf, dim=0, out=self.acc)


def time_indexer_steps(st, steps, flush, stream):
    """Event-timed indexer steps, L2 flushed before each; per chunk: the
    schedule launch (chunks of more than 256 units), then either the logits and
    top-k launches or (st.fused) the one fused score + top-k launch.  Returns
    per-step lists of ms: "step" from a pass with events around each whole step
    only (so nothing sits between the launches of a step: the top-k launches as
    a programmatic dependent of the logits kernel), the per-kernel times from a
    second pass with events between the launches ("logits" is the fused launch
    when fused, "topk" 0)."""
    from deepseek_sparse_attention_mqa_gb300 import _abi
    c = st.case
    chunks = [(rb, re) for rb, re in st.chunks if re > rb]
    nck = len(chunks)
    whole = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s in range(steps):
        flush(s)
        whole[s][0].record(stream)
        st.run()
        whole[s][1].record(stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 * nck + 1)] for _ in range(steps)]
    for s in range(steps):
        flush(s)
        e = ev[s]
        e[0].record(stream)
        for ci, (rb, re) in enumerate(chunks):
            inline = st.inline[(rb, re)]          # no schedule launch: the logits kernel builds the units
            if not inline:
                _abi.build_schedule(c.context_lens, c.batch, c.next_n, c.num_heads, rb, re, st.sched, st.status,
                                    compress_ratio=st.ratio)
            e[3 * ci + 1].record(stream)
            if st.fused:
                _abi.score_topk(c.q, c.q_scales, c.fmt, c.weights, c.num_heads, st.kcache, c.context_lens,
                                c.batch, c.next_n, rb, re, None if inline else st.sched, st.logits, st.width,
                                c.topk, st.idx[rb:re], st.count[rb:re], st.fused_ws, st.status)
                e[3 * ci + 2].record(stream)
            else:
                _abi.mqa_logits(c.q, c.q_scales, c.fmt, c.weights, c.num_heads, st.kcache, c.context_lens,
                                c.batch, c.next_n, rb, re, None if inline else st.sched, st.logits, st.width,
                                st.status)
                e[3 * ci + 2].record(stream)
                st.topk_chunk(rb, re)
            e[3 * ci + 3].record(stream)
    torch.cuda.synchronize()
    return {
        "step": [w[0].elapsed_time(w[1]) for w in whole],
        "step_with_kernel_events": [e[0].elapsed_time(e[-1]) for e in ev],
        "schedule": [sum((e[3 * ci] if ci else e[0]).elapsed_time(e[3 * ci + 1]) for ci in range(nck)) for e in ev],
        "logits": [sum(e[3 * ci + 1].elapsed_time(e[3 * ci + 2]) for ci in range(nck)) for e in ev],
        "topk": [sum(e[3 * ci + 2].elapsed_time(e[3 * ci + 3]) for ci in range(nck)) for e in ev],
        "chunks": nck,
    }


def kernel_ms_summary(t, fused, extra=None):
    d = {"schedule": round(statistics.mean(t["schedule"]), 5), "chunks": t["chunks"]}
    if fused:
        d["score_topk"] = round(statistics.mean(t["logits"]), 5)
    else:
        d["logits"] = round(statistics.mean(t["logits"]), 5)
        d["topk"] = round(statistics.mean(t["topk"]), 5)
    d.update(extra or {})
    return d


def logits_roofline(case, workload, logits_ms_per_launch, nck, fused=False):
    """Roofline of the logits kernel (fused: the score + top-k kernel): HBM
    bytes for the decode-type workloads (the fused kernel also writes the index
    rows), FP8 tensor flops for the prefill (compute-bound) workload."""
    from deepseek_sparse_attention_mqa_gb300 import inputs
    hbm, bf16, _, src = measured_peaks()
    pairs = scored_pairs(case)
    base = "logits_fp8" if case.fmt == inputs.FMT_FP8 else "logits_mxfp4"
    kname = base + (" + fused top-k (indexer_score_topk)" if fused else " (indexer_mqa_logits_paged)")
    tkey = base + ("_fused" if fused else "")
    if workload == "prefill":
        # FP8 MMA work per launch (one chunk): 2 * pairs * heads * head_dim
        flops = 2.0 * pairs * case.num_heads * case.head_dim / nck
        achieved = flops / (logits_ms_per_launch * 1e-3) / 1e12
        fp8_peak = 2.0 * bf16                             # nominal fp8 : bf16 = 2 : 1
        return {"kernel": kname + ", per chunk launch", "bound": "tensor",
                "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / fp8_peak, 4),
                "peak_source": src + " bf16 burst x 2 (nominal fp8/bf16 ratio)",
                "algorithmic_flops": flops, "traffic": load_traffic(tkey, workload)}
    lg_bytes = (logits_algorithmic_bytes(case) + (case.rows * case.topk * 4 if fused else 0)) / nck
    achieved = lg_bytes / (logits_ms_per_launch * 1e-3) / 1e9
    return {"kernel": kname, "bound": "hbm",
            "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_source": src,
            "algorithmic_bytes": lg_bytes, "traffic": load_traffic(tkey, workload)}


def measure_indexer_config(workload, dev, steps, flush, fused=True, case=None):
    """One indexer configuration timed on its own: the configuration's value,
    per-kernel times and the roofline of its dominant kernel."""
    from deepseek_sparse_attention_mqa_gb300 import inputs
    from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep
    own = case is None
    if own:
        case = inputs.make_case(workload, device=dev)
    st = SparseAttentionStep(case, with_mla=False, fused=fused)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    status = st.device_status()
    t = time_indexer_steps(st, steps, flush, stream)
    pairs = scored_pairs(case)
    ms = statistics.mean(t["step"])
    nck = t["chunks"]
    res = {"workload": WORKLOADS.get(workload, workload), "fused": fused,
           "value": round(pairs / (ms * 1e-3) / 1e3, 1), "unit": UNIT,
           "ms_per_step": round(ms, 5), "steps": steps, "scored_pairs_per_step": pairs,
           "kernel_ms": kernel_ms_summary(t, fused),
           "roofline": logits_roofline(case, workload, statistics.mean(t["logits"]) / nck, nck, fused),
           "gpu_launches_per_step": st.launches_per_step(), "device_status": status}
    del st
    if own:
        del case
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs
    from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(_abi.LIB_PATH):
        build.build()
    if world > 1:
        torch.distributed.barrier()
    _abi.lib()

    case = inputs.make_case(args.workload, device=dev)
    fused = args.fused
    st = SparseAttentionStep(case, with_mla=False, fused=fused)
    pairs = scored_pairs(case)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    status = st.device_status()
    if status != 0:
        raise RuntimeError("device status %#x after warm-up" % status)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    t = time_indexer_steps(st, args.steps, flush, stream)
    t_end = time.time()
    if world > 1:
        torch.distributed.barrier()
    nck = t["chunks"]
    total_ms = max_over_ranks(sum(t["step"]), world, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_value(pairs, world, ms_per_step)

    clocks = sampler.summary(t_begin, t_end) if sampler else None
    if sampler:
        sampler.stop()

    result = None
    if rank == 0:
        n_side = max(10, min(200, args.steps))
        # the same steps with the former flush (a 1 GiB WRITE), once, for comparison:
        # its dirty lines are written back inside the timed kernel
        wbuf = torch.empty(int(2 ** 30) // 4, dtype=torch.float32, device=dev)
        tw = time_indexer_steps(st, n_side, lambda s: wbuf.fill_(float(s)), stream)
        del wbuf
        e2e = measure_e2e(st, case, args, pairs, dev)
        roof = logits_roofline(case, args.workload, statistics.mean(t["logits"]) / nck, nck, fused)
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if case.fmt == inputs.FMT_FP8 else "e2m1", "data": "synthetic",
            "config": {"workload": WORKLOADS.get(args.workload, args.workload), "batch": case.batch,
                       "next_n": case.next_n, "heads": case.num_heads, "head_dim": case.head_dim,
                       "page_kv": case.page_kv, "topk": case.topk, "scored_pairs_per_step": pairs,
                       "seed": case.meta["seed"], "l2": "flushed between steps (384 MiB read)",
                       "parallelism": "replicas"},
            "kernel_ms": kernel_ms_summary(t, fused, {"first_kernel_after_write_flush":
                                                      round(statistics.mean(tw["logits"]), 5),
                                                      "step_with_kernel_events":
                                                      round(statistics.mean(t["step_with_kernel_events"]), 5)}),
            "fused_score_topk": fused,
            "roofline": roof,
            "gpu_launches": st.launches_per_step() * args.steps,
            "clocks": clocks,
            "e2e": e2e,
        }
        # the same workload with the other top-k arrangement (separate launches
        # when the headline is fused, and vice versa)
        result["unfused" if fused else "fused"] = measure_indexer_config(args.workload, dev, n_side, flush,
                                                                         not fused, case)
        if args.workload == "decode" and not args.skip_configs:
            result["spec_mxfp4"] = measure_indexer_config("spec_mxfp4", dev, n_side, flush, fused)
            result["prefill"] = measure_indexer_config("prefill", dev, max(5, min(20, args.steps)), flush,
                                                       False)
        if not args.skip_configs:
            result["kv_scatter"] = measure_scatter(dev, flush, n_side)
        if not args.skip_full_step:
            result["full_step"] = measure_full_step(dev, args, flush, fused=fused)
            result["full_step_indexer_h64"] = measure_full_step(dev, args, flush, "full_step_h64", fused=fused)
        if not args.skip_cpu:
            result["cpu_baseline"] = cpu_baseline(case, pairs)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result


def load_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from one ncu
    capture (profiles/traffic.json), or None when there is none or the kernel's
    sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get("%s/%s" % (kernel, workload))
    if not d:
        return None
    h = hashlib.sha256()
    for name in d["source_files"]:
        with open(os.path.join(ROOT, "deepseek_sparse_attention_mqa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != d["source_sha256_16"]:
        return None
    return d["traffic_bytes_per_launch"]


def measure_e2e(st, case, args, pairs, dev):
    """Same metric through the step API with host buffers, the way a serving
    loop runs it: every step copies its query-side inputs (one packed pinned
    arena: q, weights, context lengths, block table) to the device, runs, and
    reads its top-k indices back to pinned host memory.  HostStepPipeline
    overlaps step i's computation with the input copy of step i + 1 and the
    result copy of step i - 1 (two slots, three streams); the timed region runs
    from before the first input copy to after the last result copy.  L2 is not
    flushed inside it: a decode step streams more K pages (~152 MB) than L2
    holds.  The serial figure (copy in, run, copy out, one step at a time, L2
    evicted before each) is reported beside it."""
    from deepseek_sparse_attention_mqa_gb300.step import HostStepPipeline, SparseAttentionStep, StepInputs
    steps = max(20, args.steps // 2)
    # serial: one step at a time
    ins = StepInputs(case, with_mla=False)
    sst = SparseAttentionStep(ins.case(), with_mla=False, fused=st.fused)
    idx_host = torch.empty(sst.idx.shape, dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream()
    for _ in range(3):
        ins.copy_in(stream)
        sst.run()
        idx_host.copy_(sst.idx, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    flush = L2Flush(dev)
    tot = 0.0
    n_serial = max(10, steps // 2)
    for s in range(n_serial):
        flush(s)
        e0.record(stream)
        ins.copy_in(stream)
        sst.run()
        idx_host.copy_(sst.idx, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    ms_serial = tot / n_serial
    del sst, ins
    # pipelined
    pipe = HostStepPipeline(case, with_mla=False, fused=st.fused)
    for _ in range(4):
        pipe.submit()
    pipe.synchronize()
    torch.cuda.synchronize()
    e0.record(pipe.h2d_stream)
    c0 = time.perf_counter()
    for _ in range(steps):
        pipe.submit()
    host_us = (time.perf_counter() - c0) * 1e6 / steps
    e1.record(pipe.d2h_stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    res = {"value": round(pairs / (ms * 1e-3) / 1e3, 1), "unit": UNIT, "ms_per_step": round(ms, 5),
           "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes, "steps": steps,
           "mode": "pipelined host I/O (HostStepPipeline: two slots, each step's computation one CUDA-graph "
                   "replay; copies overlap the previous and next steps' computation)",
           "host_submit_us_per_step": round(host_us, 1),
           "l2": "not flushed between steps: each step reads ~152 MB of K pages, more than the 126 MB L2",
           "serial": {"value": round(pairs / (ms_serial * 1e-3) / 1e3, 1), "ms_per_step": round(ms_serial, 5),
                      "steps": n_serial}}
    del pipe
    # the same loop with the two slots computing on their own streams, as for two
    # independent batches (consecutive steps of one batch depend on each other)
    pipe = HostStepPipeline(case, with_mla=False, fused=st.fused, overlap_steps=True)
    for _ in range(4):
        pipe.submit()
    pipe.synchronize()
    torch.cuda.synchronize()
    e0.record(pipe.h2d_stream)
    for _ in range(steps):
        pipe.submit()
    e1.record(pipe.d2h_stream)
    e1.synchronize()
    ms_ov = e0.elapsed_time(e1) / steps
    res["independent_batches_overlapped"] = {"value": round(pairs / (ms_ov * 1e-3) / 1e3, 1),
                                             "ms_per_step": round(ms_ov, 5), "steps": steps}
    del pipe
    return res


def measure_full_step(dev, args, flush, workload="full_step", fused=True):
    """Full decode step (indexer, top-k, sparse MLA 128 heads 576/512 on an FP8
    latent, lens U[8192,131072], top-k 2048) captured in one CUDA graph; us/step
    over replays, L2 flushed.  Also times each stage alone (eager launches,
    events on the launching stream)."""
    from deepseek_sparse_attention_mqa_gb300 import inputs
    from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep
    case = inputs.make_case(workload, device=dev)
    torch.cuda.empty_cache()             # drop the generator's temporaries (the latent pool is built in fp32)
    st = SparseAttentionStep(case, with_mla=True, fused=fused)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            st.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    stream = torch.cuda.current_stream()
    times = []
    n = max(20, min(200, args.steps // 10))
    for i in range(n + 3):
        flush(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e3)
    # per-stage device time, eager (one chunk: decode rows fit the logits budget)
    stage = {"indexer": [], "topk": [], "mla": []} if not fused else {"score_topk": [], "mla": []}
    (rb, re), = [(a, b) for a, b in st.chunks if b > a]
    for i in range(n):
        flush(i)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        if fused:
            st.score_topk_chunk(rb, re)
            ev[1].record(stream)
            ev[2].record(stream)
        else:
            st.indexer_chunk(rb, re)
            ev[1].record(stream)
            st.topk_chunk(rb, re)
            ev[2].record(stream)
        st.mla()
        ev[3].record(stream)
        ev[3].synchronize()
        if fused:
            stage["score_topk"].append(ev[0].elapsed_time(ev[1]) * 1e3)
        else:
            stage["indexer"].append(ev[0].elapsed_time(ev[1]) * 1e3)
            stage["topk"].append(ev[1].elapsed_time(ev[2]) * 1e3)
        stage["mla"].append(ev[2].elapsed_time(ev[3]) * 1e3)
    status = st.device_status()
    # sparse MLA tensor work: QK^T over d_qk and PV over d_v for every (row, head, selected token)
    mla_us = statistics.median(stage["mla"])
    mla_flops = 2.0 * case.rows * case.mla_heads * case.topk * (case.d_qk + case.d_v)
    _, bf16, _, src = measured_peaks()
    return {"workload": "full sparse-attention decode step: batch 64, indexer %d heads x %d FP8 page 64, "
                        "lens U[8192,131072], top-k 2048, sparse MLA 128 heads q/k 576 v 512 FP8 latent"
                        % (case.num_heads, case.head_dim), "fused_score_topk": fused,
            "us_per_step_median": round(statistics.median(times), 2),
            "us_per_step_mean": round(statistics.mean(times), 2), "replays": n,
            "stage_us_median": {k: round(statistics.median(v), 2) for k, v in stage.items()},
            "mla_roofline": {"bound": "tensor", "achieved": round(mla_flops / (mla_us * 1e-6) / 1e12, 1),
                             "peak": bf16, "unit": "TFLOP/s", "frac": round(mla_flops / (mla_us * 1e-6) / 1e12 / bf16, 4),
                             "peak_source": src + " bf16 burst (f16 operands run at the bf16 rate)",
                             "algorithmic_flops": mla_flops,
                             "traffic": load_traffic("sparse_mla_tc", "full_step") if workload == "full_step" else None},
            "launches_per_step": st.launches_per_step(), "device_status": status}


def measure_scatter(dev, flush, steps):
    """K-cache quantise/scatter of one prefill's and one decode step's new tokens
    (bf16 K, 128 dims) into a shuffled page-64 FP8 cache and a page-32 MXFP4
    cache; HBM roofline on the algorithmic bytes (K read once, codes + scales
    written once, slot mapping read once)."""
    from deepseek_sparse_attention_mqa_gb300 import _abi
    hbm, _, _, src = measured_peaks()
    out = {}
    for name, n, fmt, P in (("prefill_fp8", 16384, 0, 64), ("prefill_mxfp4", 16384, 1, 32),
                            ("decode_fp8", 64, 0, 64)):
        D = 128
        g = torch.Generator(device=dev).manual_seed(7)
        pages = 2 * ((n + P - 1) // P)
        tok = D if fmt == 0 else D // 2
        stok = 4 if fmt == 0 else D // 32
        vals = torch.zeros((pages, P * tok), dtype=torch.uint8, device=dev)
        scs = torch.zeros((pages, P * stok + (16 if fmt == 1 else 0)), dtype=torch.uint8, device=dev)
        bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
        cache = _abi.make_cache(fmt, D, P, pages, vals, P * tok, tok, scs, scs.shape[1], stok, bt)
        k = torch.randn((n, D), generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(pages * P, generator=g, device=dev)[:n].to(torch.int64)
        stream = torch.cuda.current_stream()
        for _ in range(3):
            _abi.kv_quantize_scatter(k, slots, cache)
        ts = []
        for i in range(steps):
            flush(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _abi.kv_quantize_scatter(k, slots, cache)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ts)
        nbytes = n * (D * 2 + tok + stok + 8)
        out[name] = {"tokens": n, "head_dim": D, "format": "e4m3 + fp32 token scale" if fmt == 0 else "MXFP4",
                     "page_kv": P, "us_median": round(us, 2),
                     "roofline": {"bound": "hbm", "achieved": round(nbytes / (us * 1e-6) / 1e9, 1), "peak": hbm,
                                  "unit": "GB/s", "frac": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4),
                                  "peak_source": src, "algorithmic_bytes": nbytes}}
    return out


def cpu_baseline(case, pairs, mac_budget=12e9):
    """fp64 oracle (logits + full-sort top-k) on the host cores over a bounded,
    contiguous block of rows of the same workload (all rows when they fit the
    multiply-accumulate budget, ~10-30 s of CPU work)."""
    import oracle
    from oracle.cases import oracle_cache, visible
    per_pair = case.num_heads * case.head_dim
    vis = [visible(case, r) for r in range(case.rows)]
    if sum(vis) * per_pair <= mac_budget:
        rb, re = 0, case.rows
    else:
        mid = case.rows // 2
        rb = re = mid
        acc = 0
        while re < case.rows and acc + vis[re] * per_pair <= mac_budget:
            acc += vis[re] * per_pair
            re += 1
        re = max(re, rb + 1)
    cache, _ = oracle_cache(case.kcache, case.block_table)
    ctx = case.context_lens.cpu()
    t0 = time.time()
    if case.q_scales is None:
        lg = oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), cache, ctx, case.next_n, rb, re,
                               width=case.width)
    else:
        lg = oracle.logits_mxfp4(case.q.cpu(), case.q_scales.cpu(), case.weights.cpu(), cache, ctx,
                                 case.next_n, rb, re, width=case.width)
    oracle.topk(lg, ctx, case.next_n, case.topk, rb, re)
    dt = time.time() - t0
    sp = sum(vis[rb:re])
    return {"value": round(sp / dt / 1e3, 2), "unit": UNIT, "cores": oracle.threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "rows [%d, %d) of %d of the same workload (%d scored pairs): fp64 logits + "
                      "full-sort top-k" % (rb, re, case.rows, sp)}


def run_reference(args, rank, world):
    """The oracle timed as the reference arm, on the same workload and metric.
    Each step scores one row of the workload over at most its first 4096 visible
    tokens (rows taken in turn), so that K steps stay within minutes."""
    if rank != 0:
        return None
    import oracle
    from deepseek_sparse_attention_mqa_gb300 import inputs
    from oracle.cases import oracle_cache
    oracle.build()
    case = inputs.make_case(args.workload, device="cpu")
    cache, _ = oracle_cache(case.kcache, case.block_table)
    q, w = case.q, case.weights
    n = case.next_n
    cap = 4096
    times, pairs_tot = [], 0
    for s in range(args.warmup + args.steps):
        r = s % case.rows
        b = r // n
        L = min(int(case.context_lens[b]), cap)
        ctx = torch.tensor([L], dtype=torch.int32)
        bt_cache = oracle.PagedBytes(cache.values, cache.vps, cache.vts, cache.scales, cache.sps,
                                     cache.sts, cache.block_table[b:b + 1], cache.page_kv,
                                     cache.num_pages)
        t0 = time.time()
        lg = oracle.logits_fp8(q[b * n:(b + 1) * n], w[b * n:(b + 1) * n], bt_cache, ctx, n,
                               width=L)
        oracle.topk(lg, ctx, n, case.topk)
        dt = time.time() - t0
        if s >= args.warmup:
            times.append(dt)
            pairs_tot += sum(oracle.visible(L, n, i) for i in range(n))
    tot = sum(times)
    v = pairs_tot / tot / 1e3
    ms = tot / len(times) * 1e3
    return {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "sample": "per step one sequence's rows over its first <= %d tokens" % cap},
            "cpu_baseline": {"value": round(v, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "per step one sequence (rows in turn) over its first <= %d "
                                       "visible tokens: fp64 logits + full-sort top-k" % cap},
            "e2e": {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-full-step", action="store_true")
    ap.add_argument("--skip-configs", action="store_true")
    ap.add_argument("--fused", action="store_true",
                    help="headline step with the fused score + top-k launch")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
