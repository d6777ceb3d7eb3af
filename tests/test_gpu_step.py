"""Whole sparse-attention step on the GPU: CUDA-graph capture with context
lengths changing between replays (the schedule is rebuilt on the device inside
the graph every replay), and the full-size decode step checked on sampled rows."""
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


def check_indexer_rows(case, st, rows, ctx_cpu):
    cache, seqs = parity.oracle_cache(case.kcache, case.block_table, seqs=sorted({r // case.next_n for r in rows}))
    pos = {b: j for j, b in enumerate(seqs)}
    lg = st.logits.cpu().numpy() if st.rows_per_chunk >= case.rows else None
    idx = st.idx.cpu().numpy()
    for r in rows:
        b, i = divmod(r, case.next_n)
        sub_ctx = np.zeros(len(seqs), np.int32)
        sub_ctx[pos[b]] = ctx_cpu[b]
        q = case.q.cpu()[b * case.next_n:(b + 1) * case.next_n]
        w = case.weights.cpu()[b * case.next_n:(b + 1) * case.next_n]
        # put this sequence's rows at sub-batch position pos[b]
        qq = torch.zeros((len(seqs) * case.next_n,) + tuple(q.shape[1:]), dtype=q.dtype)
        ww = torch.zeros((len(seqs) * case.next_n, w.shape[1]), dtype=w.dtype)
        qq[pos[b] * case.next_n:(pos[b] + 1) * case.next_n] = q
        ww[pos[b] * case.next_n:(pos[b] + 1) * case.next_n] = w
        rr = pos[b] * case.next_n + i
        o = oracle.logits_fp8(qq, ww, cache, sub_ctx, case.next_n, rr, rr + 1, width=case.width)[0]
        vis = oracle.visible(int(ctx_cpu[b]), case.next_n, i)
        if lg is not None:
            parity.check_logits([lg[r]], [o], [vis])
        scale = float(np.max(np.abs(o[:vis]))) if vis else 1.0
        parity.check_topk_tolerant(idx[r:r + 1], [o], [vis], case.topk, scale)


def test_graph_replay_with_changing_lengths():
    lens = [1000, 2000, 1500, 64, 3000, 1]
    case = inputs.make_case("decode", device="cuda", lens=lens, num_heads=64, width=3000,
                            topk=512, seed=41)
    st = SparseAttentionStep(case, with_mla=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st.run()
    torch.cuda.synchronize()
    for new in ([1000, 2000, 1500, 64, 3000, 1], [10, 1999, 700, 0, 2900, 1],
                [1000, 128, 1500, 64, 129, 1]):
        case.context_lens.copy_(torch.tensor(new, dtype=torch.int32))
        st.logits.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert st.device_status() == 0
        check_indexer_rows(case, st, list(range(case.rows)), np.array(new, np.int32))


def check_mla_rows(case, st, rows):
    """MLA output of sampled rows on the GPU's own top-k selection vs the oracle."""
    cache, _ = parity.oracle_cache(case.latent, case.block_table, seqs=rows)
    idx = st.idx.cpu().numpy()
    for j, r in enumerate(rows):
        o, l = oracle.sparse_mla(case.q_mla[r:r + 1].cpu(), case.softmax_scale, oracle.FMT_FP8,
                                 cache, idx[r:r + 1], case.d_v, seq_of_row=[j])
        parity.check_mla(st.out[r:r + 1], st.lse[r:r + 1], o, l)


def test_full_step_graph_with_mla_replayed_with_changing_lengths():
    """The full decode step at full size (indexer 4 heads x 32, lens up to
    131072, top-k 2048, sparse MLA 128 heads 576/512 on the FP8 latent) captured
    once in ONE CUDA graph with the MLA stage, then replayed after the context
    lengths change: every replay recomputes the work from the new lengths (no
    stale windows), and sampled rows' logits, top-k and MLA output match the
    oracle.  The new lengths include an empty history, rows shorter than k and
    rows exactly at k."""
    case = inputs.make_case("full_step", device="cuda")
    st = SparseAttentionStep(case, with_mla=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st.run()
    torch.cuda.synchronize()
    orig = case.context_lens.cpu().numpy().copy()
    shrunk = orig // 2
    shrunk[:6] = [0, 1, 2047, 2048, 2049, 8192]
    rows = [0, 1, 2, 3, 4, 5, 31, 63]
    for new in (orig, shrunk, orig):
        case.context_lens.copy_(torch.from_numpy(np.ascontiguousarray(new, np.int32)))
        st.logits.fill_(float("nan"))
        st.out.fill_(float("nan"))
        st.idx.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert st.device_status() == 0
        check_indexer_rows(case, st, rows, new)
        check_mla_rows(case, st, rows)


def test_full_step_full_size_sampled_rows():
    case = inputs.make_case("full_step", device="cuda")
    st = SparseAttentionStep(case, with_mla=True)
    st.run()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    rows = [3, 50]
    check_indexer_rows(case, st, rows, case.context_lens.cpu().numpy())
    # MLA on the GPU's own selection
    cache, seqs = parity.oracle_cache(case.latent, case.block_table, seqs=rows)
    idx = st.idx.cpu().numpy()
    for j, r in enumerate(rows):
        o, l = oracle.sparse_mla(case.q_mla[r:r + 1].cpu(), case.softmax_scale, oracle.FMT_FP8,
                                 cache, idx[r:r + 1], case.d_v, seq_of_row=[j])
        parity.check_mla(st.out[r:r + 1], st.lse[r:r + 1], o, l)


@pytest.mark.parametrize("overlap", [False, True])
def test_host_pipeline_matches_the_step_and_the_oracle(overlap):
    """HostStepPipeline (inputs from pinned host memory, copies overlapping the
    neighbouring steps' computation; with overlap, the two slots' computations
    overlap too): slot 1 is given other context lengths
    than slot 0, several steps run back to back, and every step's top-k indices
    on the host equal those of the plain step on the same inputs; sampled rows
    of the shorter-length slot also match the oracle."""
    import dataclasses
    from deepseek_sparse_attention_mqa_gb300.step import HostStepPipeline
    case = inputs.make_case("decode", device="cuda")
    orig = case.context_lens.cpu().numpy().copy()
    shrunk = orig // 3
    shrunk[:4] = [0, 1, 2047, 2048]
    refs = []
    for lens in (orig, shrunk):
        c = dataclasses.replace(case, context_lens=torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda())
        st = SparseAttentionStep(c, with_mla=False)
        st.run()
        torch.cuda.synchronize()
        refs.append((st.idx.cpu().numpy(), st))
    pipe = HostStepPipeline(case, overlap_steps=overlap)
    pipe.inputs[1].host["context_lens"].copy_(torch.from_numpy(np.ascontiguousarray(shrunk, np.int32)))
    for it in range(6):
        slot = pipe.submit()
        if it >= 1:
            prev = slot ^ 1
            got = pipe.results(prev).numpy()
            assert np.array_equal(np.sort(got, axis=1), np.sort(refs[prev][0], axis=1)), "slot %d" % prev
    pipe.synchronize()
    for s in (0, 1):
        assert np.array_equal(np.sort(pipe.results(s).numpy(), axis=1), np.sort(refs[s][0], axis=1))
        assert pipe.steps[s].device_status() == 0
    check_indexer_rows(dataclasses.replace(case, context_lens=refs[1][1].case.context_lens), refs[1][1],
                       [0, 1, 2, 3, 17], shrunk)
