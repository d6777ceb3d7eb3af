"""GPU parity of the per-row top-k (libdsa radix select) against the oracle's
full sort: bit-exact index sets on identical logits (ties -> lower position),
and the tolerance rule end to end on the indexer's own logits."""
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


def run_topk(logits, lens, next_n, k, width):
    dev = torch.device("cuda")
    lg = logits.to(dev)
    ctx = torch.tensor(lens, dtype=torch.int32, device=dev)
    rows = len(lens) * next_n
    idx = torch.full((rows, k + 3), 12345, dtype=torch.int32, device=dev)
    cnt = torch.empty((rows,), dtype=torch.int32, device=dev)
    st = torch.zeros((1,), dtype=torch.int32, device=dev)
    _abi.topk(lg, width, ctx, len(lens), next_n, 0, rows, k, idx, cnt, None, st)
    torch.cuda.synchronize()
    out = idx.cpu().numpy()
    assert np.all(out[:, k:] == 12345), "wrote past k"
    return out[:, :k], cnt.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("width,k", [(4096, 64), (32768, 2048), (65536, 512), (100000, 2048)])
def test_same_logits_exact(width, k):
    g = torch.Generator().manual_seed(width + k)
    lens = [0, 1, k - 1, k, k + 1, width // 3, width]
    rows = torch.randn((len(lens), width), generator=g)
    rows[3, :] = torch.round(rows[3, :] * 2)          # many exact ties
    rows[5, : width // 3] = 1.5                         # all equal
    rows[6, ::2] = -0.0                                  # signed zeros tie with +0
    rows[6, 1::2] = 0.0
    idx, cnt, st = run_topk(rows, lens, 1, k, width)
    assert st == 0
    ref_idx, ref_cnt = oracle.topk(rows.double().numpy(), lens, 1, k)
    assert list(cnt) == list(ref_cnt)
    parity.check_topk_same_input(idx, ref_idx, lens, k)
    # ties resolve to the lower positions: the all-equal row takes 0..k-1
    assert sorted(idx[5].tolist()) == list(range(k))


def topk_cluster_size(rows, width, sm_count):
    """The cluster size the library's top-k launch picks (CTAs per row): enough
    that the widest slice fits in shared memory, then enough to cover ~1.5x the
    SMs, at most 8."""
    C = 1
    while C < 8 and -(-width // C) > 16384:
        C *= 2
    while C < 8 and rows * C * 2 < 3 * sm_count:
        C *= 2
    return C


@pytest.mark.parametrize("rows,width,k,expect_c", [
    (64, 32768, 2048, 4),      # the decode workload's launch: 64 rows x 32768
    (256, 65536, 512, 4),      # the speculative workload's launch: 128 x 2 rows x 65536
    (320, 16384, 2048, 1),     # a prefill chunk's launch shape: >= 304 rows x 16384
    (64, 131072, 2048, 8),     # the full step's launch: 64 rows x 131072
    (160, 32768, 2048, 2),     # two CTAs per row
])
def test_workload_launch_shapes_exact(rows, width, k, expect_c):
    """Same logits on both sides at the row counts and widths the real workloads
    launch with, so the cluster sizes they run at (4 CTAs per row for decode and
    speculative decode, 1 for prefill chunks) are compared with the oracle's
    full sort: identical index sets, ties to the lower position.  Some rows put
    every key in one first-round bin (distinct values in [1, 1.25), the top 11
    key bits), so the histogram is refined in further rounds across the cluster."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert topk_cluster_size(rows, width, sms) == expect_c
    g = torch.Generator().manual_seed(rows + width + k)
    lens = torch.randint(k // 2, width + 1, (rows,), generator=g).tolist()
    lens[:6] = [0, 1, k, k + 1, width, width - 1]
    logits = torch.randn((rows, width), generator=g)
    logits[2::7] = torch.round(logits[2::7] * 4)         # rows full of exact ties
    logits[3::11, ::3] = 2.5                             # a heavy tie at the top
    logits[4::13] = 1.0 + 0.25 * torch.rand((logits[4::13].shape[0], width), generator=g)
    idx, cnt, st = run_topk(logits, lens, 1, k, width)
    assert st == 0
    ref_idx, ref_cnt = oracle.topk(logits.double().numpy(), lens, 1, k)
    assert list(cnt) == list(ref_cnt)
    parity.check_topk_same_input(idx, ref_idx, lens, k)


def test_next_n_windows():
    g = torch.Generator().manual_seed(2)
    lens = [10, 3000]
    rows = torch.randn((6, 3000), generator=g)
    idx, cnt, _ = run_topk(rows, lens, 3, 64, 3000)
    vis = [oracle.visible(L, 3, i) for L in lens for i in range(3)]
    ref_idx, _ = oracle.topk(rows.double().numpy(), lens, 3, 64)
    parity.check_topk_same_input(idx, ref_idx, vis, 64)


def test_end_to_end_on_indexer_logits():
    case = inputs.make_case("decode", device="cuda", lens=[3000, 2049, 700, 4096], num_heads=64,
                            width=4096, topk=2048, seed=21)
    st = SparseAttentionStep(case, with_mla=False)
    st.run()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    cache, _ = parity.oracle_cache(case.kcache, case.block_table)
    ref = oracle.logits_fp8(case.q.cpu(), case.weights.cpu(), cache, case.context_lens.cpu(), 1,
                            width=case.width)
    vis = [parity.visible(case, r) for r in range(case.rows)]
    scale = max(float(np.nanmax(np.abs(ref[r, :v]))) for r, v in enumerate(vis))
    parity.check_topk_tolerant(st.idx.cpu().numpy(), ref, vis, case.topk, scale)
