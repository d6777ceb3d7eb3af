"""The bounded on-chip waits: a wait whose arrival never comes (a device word
the host leaves unset) runs out after its limit, reports DSA_DEV_TIMEOUT in the
status word and returns -- the GPU context stays usable for the next call."""
import pytest
import torch

from deepseek_sparse_attention_mqa_gb300 import _abi, build, inputs
from deepseek_sparse_attention_mqa_gb300.step import SparseAttentionStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.lib()


def test_wait_runs_out_and_reports_timeout():
    dev = torch.device("cuda")
    flag = torch.zeros((1,), dtype=torch.int32, device=dev)      # never set to 1
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    _abi.wait_selftest(flag, 1, 20000, status)                   # 20 ms limit
    assert _abi.device_status(status) & _abi.DEV_TIMEOUT
    # the condition holds: the same wait completes and reports nothing
    flag.fill_(1)
    status.zero_()
    _abi.wait_selftest(flag, 1, 20000, status)
    assert _abi.device_status(status) == 0
    # the context is still usable: a regular step runs and reports nothing
    case = inputs.make_case("tiny", device=dev, with_mla=False)
    st = SparseAttentionStep(case, with_mla=False)
    st.run()
    torch.cuda.synchronize()
    assert st.device_status() == 0


def test_wait_selftest_argument_checks():
    dev = torch.device("cuda")
    flag = torch.zeros((1,), dtype=torch.int32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    for bad in (0, 3_000_000):
        with pytest.raises(_abi.DSAError) as ei:
            _abi.wait_selftest(flag, 1, bad, status)
        assert ei.value.status == _abi.DSA_ERR_INVALID_ARG
