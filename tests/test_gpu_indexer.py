"""GPU parity of the indexer schedule + paged MQA logits (libdsa, tcgen05/TMA)
against the fp64 oracle, element by element, plus device-status behaviour.

Case matrix after "SM120 FP8 paged MQA page 32" (Validation): page 32/64 x
heads 16/32/64 x next_n 1/2/3 x head_dim 32/64/128, shuffled physical pages,
padded strides, empty history, partial pages; plus heads 4/8/128, a chunked
causal prefill, and the full-size decode workload checked on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs
from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.lib()
    oracle.build()


def gpu_logits(case, rows_per_chunk=None, width=None):
    """Run schedule + logits for every chunk; returns (rows list, step)."""
    st = SparseAttentionStep(case, with_mla=False, rows_per_chunk=rows_per_chunk)
    if width is not None:
        st.width = width
    rows = []
    for rb, re in st.chunks:
        if re == rb:
            continue
        st.logits.fill_(float("nan"))
        st.indexer_chunk(rb, re)
        torch.cuda.synchronize()
        rows.extend(list(st.logits[:re - rb].cpu().numpy()))
    return rows, st


def oracle_logits(case, rows=None):
    cache, _ = parity.oracle_cache(case.kcache, case.block_table)
    ctx = case.context_lens.cpu()
    if case.fmt == inputs.FMT_FP8:
        fn = lambda rb, re: oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), cache, ctx,
                                              case.next_n, rb, re, width=case.width)
    else:
        fn = lambda rb, re: oracle.logits_mxfp4(case.q.cpu(), case.q_scales.cpu(),
                                                case.weights.cpu(), cache, ctx, case.next_n, rb,
                                                re, width=case.width)
    if rows is None:
        return list(fn(0, case.rows))
    return [fn(r, r + 1)[0] for r in rows]


def compare_all(case, rows_per_chunk=None):
    g, st = gpu_logits(case, rows_per_chunk)
    o = oracle_logits(case)
    vis = [parity.visible(case, r) for r in range(case.rows)]
    worst, tol = parity.check_logits(g, o, vis)
    for r, v in enumerate(vis):                       # nothing written past the window
        assert np.all(np.isnan(g[r][v:])), "row %d written past its visible length" % r
    assert st.device_status() == 0
    return worst, tol


def test_tiny_workload():
    case = inputs.make_case("tiny", device="cuda", with_mla=False)
    compare_all(case)


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("next_n", [1, 2, 3])
@pytest.mark.parametrize("H", [16, 32, 64])
@pytest.mark.parametrize("P", [32, 64])
def test_matrix(P, H, next_n, D):
    lens = [0, 1, 63, 64, 65, 200, 511]
    case = inputs.make_case("decode", device="cuda", lens=lens, next_n=next_n, page_kv=P,
                            num_heads=H, head_dim=D, width=600, pool_factor=2,
                            seed=1000 + P + H + next_n + D)
    compare_all(case)


@pytest.mark.parametrize("H,next_n", [(4, 1), (4, 2), (4, 3), (8, 1), (8, 2), (128, 1), (128, 3)])
def test_other_head_counts(H, next_n):
    case = inputs.make_case("decode", device="cuda", lens=[5, 130, 257, 1000], next_n=next_n,
                            num_heads=H, head_dim=32 if H <= 8 else 128, width=1024, seed=77 + H)
    compare_all(case)


def test_padded_strides():
    case = inputs.make_case("decode", device="cuda", lens=[33, 400, 129], num_heads=32,
                            head_dim=64, page_kv=32, width=512, val_pad=512, sc_pad=64, seed=5)
    assert case.kcache.val_page_stride == 32 * 64 + 512
    compare_all(case)


def test_prefill_chunked_causal():
    T = 700
    case = inputs.make_case("prefill", device="cuda", lens=[T], next_n=T, width=T, seed=3)
    compare_all(case, rows_per_chunk=256)            # chunks 256 + 256 + 188 rows


def test_schedule_buffer_contents():
    case = inputs.make_case("decode", device="cuda", lens=[0, 129, 5000, 128], next_n=2,
                            num_heads=64, width=5000, seed=9)
    st = SparseAttentionStep(case, with_mla=False, inline_schedule=False)
    st.indexer_chunk(0, case.rows)
    torch.cuda.synchronize()
    s = st.sched.cpu().numpy()
    assert s[0] == 0x44534132 and s[1] == 4 and s[2] == 2 and s[3] == 0 and s[4] == 8
    # 32-byte records: first_row, nrows, seq, tile_begin, tile_end, vis_max, ctx_len, 0
    units = s[8:8 + 32].reshape(4, 8)
    vis = [parity.visible(case, 2 * b + 1) for b in range(4)]
    tiles = [(v + 127) // 128 for v in vis]
    begins = list(np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    assert list(units[:, 0]) == [0, 2, 4, 6] and list(units[:, 1]) == [2] * 4
    assert list(units[:, 2]) == [0, 1, 2, 3]
    assert list(units[:, 3]) == begins
    assert list(units[:, 4]) == [b + t for b, t in zip(begins, tiles)]
    assert list(units[:, 5]) == vis
    assert list(units[:, 6]) == [0, 129, 5000, 128] and list(units[:, 7]) == [0] * 4
    assert s[6] == sum(tiles)


def test_schedule_reused_across_launches():
    """One schedule, several stream-ordered logits launches (a captured decode
    graph replays the logits launch on the buffer its schedule launch filled):
    every launch reads the schedule only and reproduces the first one's logits
    bit for bit."""
    for fmt_case in ("decode", "spec_mxfp4"):
        case = inputs.make_case(fmt_case, device="cuda", batch=9, seed=21)
        st = SparseAttentionStep(case, with_mla=False, inline_schedule=False)
        st.indexer_chunk(0, case.rows)
        torch.cuda.synchronize()
        first = st.logits.clone()
        c = case
        for rep in range(3):
            st.logits.fill_(float("nan"))
            _abi.mqa_logits(c.q, c.q_scales, c.fmt, c.weights, c.num_heads, st.kcache, c.context_lens,
                            c.batch, c.next_n, 0, c.rows, st.sched, st.logits, st.width, st.status)
            torch.cuda.synchronize()
            assert st.device_status() == 0
            for r in range(c.rows):
                v = parity.visible(case, r)
                assert torch.equal(st.logits[r, :v], first[r, :v]), (fmt_case, rep, r)


@pytest.mark.parametrize("name,over", [
    ("decode", dict(lens=[0, 1, 127, 128, 129, 4000, 70], width=4000)),
    ("decode", dict(lens=[5, 300, 2049], next_n=3, num_heads=16, head_dim=64, page_kv=32, width=2100)),
    ("decode", dict(lens=[900, 33], next_n=3, num_heads=128, width=900)),
    ("decode", dict(batch=256, width=32768)),
    ("spec_mxfp4", dict(batch=40)),
])
def test_inline_schedule_matches_prebuilt(name, over):
    """Without a schedule buffer the logits kernel builds its units itself (one
    launch instead of two); the logits are bit-identical to a launch on a
    schedule built by the schedule kernel, up to the 256-unit limit."""
    case = inputs.make_case(name, device="cuda", seed=41, with_mla=False, **over)
    ref = SparseAttentionStep(case, with_mla=False, inline_schedule=False)
    got = SparseAttentionStep(case, with_mla=False)
    assert all(got.inline.values()) and not any(ref.inline.values())
    assert got.launches_per_step() == 2 and ref.launches_per_step() == 3
    for st in (ref, got):
        st.logits.fill_(float("nan"))
        st.indexer_chunk(0, case.rows)
    torch.cuda.synchronize()
    assert ref.device_status() == 0 and got.device_status() == 0
    for r in range(case.rows):
        v = parity.visible(case, r)
        assert torch.equal(ref.logits[r, :v], got.logits[r, :v]), r
        assert torch.isnan(got.logits[r, v:]).all(), r


def test_packed_step_inputs_match():
    """The packed input arena (one host-to-device copy per step) feeds the same
    kernels with the same bytes: logits and top-k are bit-identical to a step
    over the separately allocated tensors, also after the host side is
    rewritten and copied in again."""
    from deepseek_sparse_attention_mqa_gb300.step import StepInputs
    for name in ("decode", "spec_mxfp4"):
        case = inputs.make_case(name, device="cuda", batch=6, seed=5, with_mla=False)
        st = SparseAttentionStep(case, with_mla=False)
        st.run()
        ins = StepInputs(case, with_mla=False)
        st2 = SparseAttentionStep(ins.case(), with_mla=False)
        for w in ins.host["weights"], ins.device["weights"]:
            assert w.shape == case.weights.shape
        ins.host["weights"].mul_(2.0)                     # a new step's inputs ...
        ins.copy_in()
        ins.host["weights"].mul_(0.5)                     # ... and back
        ins.copy_in()
        st2.run()
        torch.cuda.synchronize()
        assert st2.device_status() == 0 and st.device_status() == 0
        # the selected set is unique; its order follows the CTAs' output reservations
        assert torch.equal(st.idx.sort(dim=1).values, st2.idx.sort(dim=1).values)
        assert torch.equal(st.count, st2.count)
        for r in range(case.rows):
            v = parity.visible(case, r)
            assert torch.equal(st.logits[r, :v], st2.logits[r, :v])


def test_decode_full_size_sampled_rows():
    """The decode workload at full size in the launch configuration the bench
    times (inline schedule, 64 rows x 32768, top-k 2048 on 4-CTA clusters):
    logits and the top-k of the kernel's own logits on sampled rows."""
    case = inputs.make_case("decode", device="cuda")
    st = SparseAttentionStep(case, with_mla=False)
    assert all(st.inline.values()) and st.launches_per_step() == 2
    st.logits.fill_(float("nan"))
    st.run()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    sample = [0, 17, 40, 63]
    q = case.q.cpu()
    w = case.weights.cpu()
    ctx = case.context_lens.cpu()
    idx = st.idx.cpu().numpy()
    for r in sample:
        cache, _ = parity.oracle_cache(case.kcache, case.block_table, seqs=[r])
        o = oracle.logits_fp8(q[r:r + 1], w[r:r + 1], cache, ctx[r:r + 1], 1, width=case.width)
        vis = parity.visible(case, r)
        parity.check_logits([st.logits[r].cpu().numpy()], [o[0]], [vis])
        scale = float(np.max(np.abs(o[0, :vis])))
        parity.check_topk_tolerant(idx[r:r + 1], [o[0]], [vis], case.topk, scale)


def test_prefill_full_size_both_chunks():
    """The prefill workload at full size as the bench runs it: 16384 causal rows
    in two 8192-row chunks (2048 work units each, so a prebuilt schedule per
    chunk and persistent CTAs walking many units), logits width 16384, top-k
    2048 on 1-CTA clusters.  Sampled rows of each chunk -- its first rows, the
    rows on both sides of the chunk boundary and the last row -- are compared
    with the oracle: logits element by element, entries past the row's window
    untouched, and the top-k of the kernel's own logits."""
    case = inputs.make_case("prefill", device="cuda")
    st = SparseAttentionStep(case, with_mla=False)
    assert st.chunks == [(0, 8192), (8192, 16384)]
    assert not any(st.inline.values())
    q, w = case.q.cpu(), case.weights.cpu()
    ctx = case.context_lens.cpu()
    cache, _ = parity.oracle_cache(case.kcache, case.block_table)
    samples = [[0, 1, 127, 128, 3001, 8190, 8191], [8192, 8193, 12345, 16382, 16383]]
    for (rb, re), rows in zip(st.chunks, samples):
        st.logits.fill_(float("nan"))
        st.indexer_chunk(rb, re)
        st.topk_chunk(rb, re)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        for r in rows:
            o = oracle.logits_fp8(q, w, cache, ctx, case.next_n, r, r + 1, width=case.width)[0]
            vis = parity.visible(case, r)
            assert vis == r + 1
            g = st.logits[r - rb].cpu().numpy()
            parity.check_logits([g], [o], [vis])
            assert np.all(np.isnan(g[vis:])), "row %d written past its window" % r
            scale = float(np.max(np.abs(o[:vis])))
            parity.check_topk_tolerant(st.idx[r:r + 1].cpu().numpy(), [o], [vis], case.topk, scale)


def test_bad_block_table_entry_sets_status():
    case = inputs.make_case("decode", device="cuda", lens=[300, 300], num_heads=16, head_dim=64,
                            width=300, seed=12)
    bt = case.block_table.clone()
    bt[1, 2] = case.kcache.num_pages + 7               # out of the pool
    case.block_table = bt
    g, st = gpu_logits(case)
    assert st.device_status() & _abi.DEV_BAD_PAGE
    o = oracle_logits(case, rows=[0])
    parity.check_logits([g[0]], o, [300])              # the other sequence is untouched


def test_width_clip_sets_status():
    case = inputs.make_case("decode", device="cuda", lens=[90, 300], num_heads=16, head_dim=64,
                            width=300, seed=13)
    st = SparseAttentionStep(case, with_mla=False)
    st.logits.fill_(float("nan"))
    st.width = 128                                     # narrower than the visible length
    st.indexer_chunk(0, 2)
    torch.cuda.synchronize()
    assert st.device_status() & _abi.DEV_WIDTH
    g = st.logits.cpu().numpy()
    o = oracle_logits(case)
    parity.check_logits([g[0], g[1]], o, [90, 128])
    assert np.all(np.isnan(g[1, 128:]))


# ------------------------------------------------------------------ MXFP4

def test_mxfp4_edge_lengths_padded_strides():
    case = inputs.make_case("spec_mxfp4", device="cuda", lens=[0, 1, 2, 31, 32, 33, 64, 200, 1000],
                            width=1024, seed=51)
    assert case.kcache.val_page_stride == 32 * 32 + 1024
    compare_all(case)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("next_n", [1, 2, 3])
@pytest.mark.parametrize("H", [16, 32, 64])
@pytest.mark.parametrize("P", [32, 64])
def test_mxfp4_matrix(P, H, next_n, D):
    case = inputs.make_case("spec_mxfp4", device="cuda", lens=[0, 1, 63, 64, 65, 200, 511],
                            next_n=next_n, page_kv=P, num_heads=H, head_dim=D, width=600,
                            seed=2000 + P + H + next_n + D)
    if D == 128 and min(next_n, 256 // H) * H > 128:
        # one TMEM accumulator per 32-element block does not fit: refused on the host
        with pytest.raises(_abi.DSAError) as ei:
            gpu_logits(case)
        assert ei.value.status == _abi.DSA_ERR_UNSUPPORTED
        return
    compare_all(case)


def test_mxfp4_full_size_sampled_rows():
    case = inputs.make_case("spec_mxfp4", device="cuda")
    g, st = gpu_logits(case)
    assert st.device_status() == 0
    q, qs, w = case.q.cpu(), case.q_scales.cpu(), case.weights.cpu()
    ctx = case.context_lens.cpu()
    lens = ctx.tolist()
    sample_seqs = [0, 3, 7] + sorted(range(len(lens)), key=lambda b: -lens[b])[:2]
    for b in sample_seqs:
        cache, _ = parity.oracle_cache(case.kcache, case.block_table, seqs=[b])
        n = case.next_n
        o = oracle.logits_mxfp4(q[b * n:(b + 1) * n], qs[b * n:(b + 1) * n], w[b * n:(b + 1) * n], cache,
                                ctx[b:b + 1], n, width=case.width)
        for i in range(n):
            r = b * n + i
            parity.check_logits([g[r]], [o[i]], [parity.visible(case, r)])


def test_schedule_of_another_call_sets_status_and_writes_nothing():
    """A prebuilt schedule that does not describe the call (built for rows
    [0, 1), passed to a call over rows [0, 2)) is refused on the device:
    DSA_DEV_SCHEDULE is set and no logit is written."""
    case = inputs.make_case("decode", device="cuda", lens=[300, 400], num_heads=16, head_dim=64,
                            width=400, seed=14)
    st = SparseAttentionStep(case, with_mla=False)
    dev = torch.device("cuda")
    n = _abi.schedule_bytes(case.batch, case.next_n, case.num_heads, 0, 2)
    sched = torch.zeros(((n + 3) // 4,), dtype=torch.int32, device=dev)
    _abi.build_schedule(case.context_lens, case.batch, case.next_n, case.num_heads, 0, 1, sched, st.status)
    st.logits.fill_(float("nan"))
    _abi.mqa_logits(case.q, case.q_scales, case.fmt, case.weights, case.num_heads, st.kcache,
                    case.context_lens, case.batch, case.next_n, 0, 2, sched, st.logits, st.width, st.status)
    torch.cuda.synchronize()
    assert st.device_status() & _abi.DEV_SCHEDULE
    assert np.all(np.isnan(st.logits[:2].cpu().numpy()))


def test_mxfp4_q_block_exponents_far_apart():
    """q whose block exponents within a head differ by more than 8 (block 0 of
    every even head scaled by 2^12, block 1 of every odd head by 2^-10): the
    kernel cannot fold them into its widened q and keeps them per block; the
    logits still match the oracle, as do those of a unit whose codes are close."""
    case = inputs.make_case("spec_mxfp4", device="cuda", lens=[0, 1, 63, 200, 511, 1000],
                            width=1024, seed=52)
    qs = case.q_scales.clone().to(torch.int32)
    qs[:, 0::2, 0] += 12
    qs[:, 1::2, 1] -= 10
    assert int(qs.max()) <= 254 and int(qs.min()) >= 1
    case.q_scales = qs.to(torch.uint8)
    compare_all(case)
