"""GPU parity of the fused indexer score + top-k (indexer_score_topk): one
launch that writes the same logits as indexer_mqa_logits_paged and the same
top-k index sets as indexer_topk.  Checked three ways: the logits and index
sets against the separate launches on the same inputs (identical); the index
sets against the oracle's full sort of the kernel's own logits (identical);
and logits plus top-k against the fp64 oracle under the tolerance rule.  The
workspace counters are reused across calls and graph replays without
clearing."""
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


def run_both(case, **kw):
    sep = SparseAttentionStep(case, with_mla=False, **kw)
    fus = SparseAttentionStep(case, with_mla=False, fused=True, **kw)
    out = []
    for st in (sep, fus):
        st.logits.fill_(float("nan"))
        st.idx.fill_(-7)
        st.count.fill_(-7)
    return sep, fus


def compare_chunkwise(case, sep, fus, oracle_rows=None):
    """Run both steps chunk by chunk; per chunk compare logits bit for bit and
    index sets exactly, plus the index sets against the oracle's sort of the
    fused kernel's own logits."""
    vis = [parity.visible(case, r) for r in range(case.rows)]
    for rb, re in fus.chunks:
        if re == rb:
            continue
        sep.logits.fill_(float("nan"))
        fus.logits.fill_(float("nan"))
        sep.indexer_chunk(rb, re)
        sep.topk_chunk(rb, re)
        fus.score_topk_chunk(rb, re)
        torch.cuda.synchronize()
        assert sep.device_status() == 0 and fus.device_status() == 0
        for r in range(rb, re):
            v = min(vis[r], fus.width)
            assert torch.equal(sep.logits[r - rb, :v], fus.logits[r - rb, :v]), r
        si = np.sort(sep.idx[rb:re].cpu().numpy(), axis=1)
        fi = np.sort(fus.idx[rb:re].cpu().numpy(), axis=1)
        assert np.array_equal(si, fi)
        assert torch.equal(sep.count[rb:re], fus.count[rb:re])
        # the fused selection is the exact top-k of its own logits
        lg = fus.logits[:re - rb].double().cpu().numpy()
        ctx = case.context_lens.cpu().numpy()
        ref_idx, ref_cnt = oracle.topk(lg, ctx, case.next_n, case.topk, rb, re)
        parity.check_topk_same_input(fus.idx[rb:re].cpu().numpy(), ref_idx, vis[rb:re], case.topk)
        assert list(fus.count[rb:re].cpu().numpy()) == list(ref_cnt)


@pytest.mark.parametrize("name,over", [
    ("decode", dict(lens=[0, 1, 2047, 2048, 2049, 5000, 70, 31000], width=31000, seed=11)),
    ("decode", dict(lens=[5, 300, 2049, 0, 4100], next_n=3, num_heads=16, head_dim=64, page_kv=32,
                    width=4100, topk=256, seed=12)),
    ("decode", dict(lens=[900, 33, 2500], next_n=3, num_heads=128, width=2500, topk=512, seed=13)),
    ("decode", dict(lens=[(i * 389) % 6000 for i in range(300)], width=6000, topk=1024, seed=14)),
    ("spec_mxfp4", dict(batch=40, seed=15)),
    ("full_step", dict(batch=6, seed=16, with_mla=False)),
])
def test_fused_matches_separate_and_oracle_sort(name, over):
    over = dict(over)
    case = inputs.make_case(name, device="cuda", **over)
    sep, fus = run_both(case)
    compare_chunkwise(case, sep, fus)


def test_fused_ties_and_constant_rows():
    """Rows whose logits are all equal (weights 0) or full of exact ties: the
    lower positions win, exactly as in the full sort."""
    case = inputs.make_case("decode", device="cuda", lens=[3000, 2500, 4096], num_heads=16, head_dim=64,
                            width=4096, topk=1000, seed=17)
    case.weights[0].zero_()                          # all logits of row 0 are exactly 0
    case.weights[1] = torch.round(case.weights[1] * 4) / 4
    sep, fus = run_both(case)
    compare_chunkwise(case, sep, fus)
    fus.run()
    torch.cuda.synchronize()
    assert sorted(fus.idx[0].cpu().tolist()) == list(range(1000))


def test_fused_prefill_chunks_prebuilt_schedule():
    """Prefill rows through the prebuilt-schedule path (chunks above 256 units):
    one CTA selects several rows of a unit in turn."""
    T = 3000
    case = inputs.make_case("prefill", device="cuda", lens=[T], next_n=T, width=T, topk=512, seed=18)
    sep, fus = run_both(case, rows_per_chunk=1536)
    assert not any(fus.inline.values())
    compare_chunkwise(case, sep, fus)


def test_fused_decode_full_size_against_oracle():
    """The decode workload at full size, in the launch configuration the bench
    times: sampled rows' logits and top-k against the fp64 oracle, and every
    row's index set equal to the separate launches'."""
    case = inputs.make_case("decode", device="cuda")
    sep, fus = run_both(case)
    assert fus.launches_per_step() == 1
    compare_chunkwise(case, sep, fus)
    q, w, ctx = case.q.cpu(), case.weights.cpu(), case.context_lens.cpu()
    idx = fus.idx.cpu().numpy()
    for r in (0, 21, 63):
        cache, _ = parity.oracle_cache(case.kcache, case.block_table, seqs=[r])
        o = oracle.logits_fp8(q[r:r + 1], w[r:r + 1], cache, ctx[r:r + 1], 1, width=case.width)[0]
        vis = parity.visible(case, r)
        parity.check_logits([fus.logits[r].cpu().numpy()], [o], [vis])
        parity.check_topk_tolerant(idx[r:r + 1], [o], [vis], case.topk, float(np.max(np.abs(o[:vis]))))


def test_fused_graph_replay_reuses_workspace():
    """Captured once, replayed with changing lengths: the per-unit counters
    return to zero after every call, so every replay selects every row."""
    lens = [4000, 2000, 1500, 64, 3000, 1, 3000, 2500]          # pages allocated for these
    case = inputs.make_case("decode", device="cuda", lens=lens, num_heads=64, width=4000, topk=2048,
                            seed=19)
    st = SparseAttentionStep(case, with_mla=False, fused=True)
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
    for new in (lens, [10, 1999, 1400, 0, 2900, 1, 2049, 2048], lens):
        case.context_lens.copy_(torch.tensor(new, dtype=torch.int32))
        st.idx.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert st.device_status() == 0
        assert int(st.fused_ws.abs().sum()) == 0
        vis = [parity.visible(case, r) for r in range(case.rows)]
        lg = st.logits.double().cpu().numpy()
        ref_idx, _ = oracle.topk(lg, np.array(new, np.int32), 1, case.topk)
        parity.check_topk_same_input(st.idx.cpu().numpy(), ref_idx, vis, case.topk)
