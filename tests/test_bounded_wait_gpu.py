"""Failure detection without a GPU fault: a bounded wait of the library that
is never satisfied gives up, reports MOE_ERR_TIMEOUT through a status word
the host reads, and leaves the context usable.  The wait polls a device word
that nothing writes (moe_selftest_bounded_wait) with a small limit, so it
ends within a few milliseconds."""
import pytest
import torch

import combine_moe_route_topk_gb300 as moe
import oracle
from combine_moe_route_topk_gb300 import workloads as W
from test_parity_gpu import _compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moe_route_topk_gb300 import _build
    _build.build()


def test_wait_on_a_flag_nothing_sets_times_out_and_the_context_stays_usable():
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    moe.selftest_bounded_wait(status, polls=1 << 12)
    torch.cuda.synchronize()
    assert int(status[0]) == moe.MOE_ERR_TIMEOUT
    # the same context still runs the path and matches the oracle
    w = W.WORKLOADS["tiny"]
    gr, _, _ = _compare(w, W.make_inputs(w))
    assert gr.status == oracle.OK


def test_wait_on_a_flag_already_set_succeeds():
    status = torch.tensor([123, 1], dtype=torch.int32, device="cuda")
    moe.selftest_bounded_wait(status, polls=1 << 12)
    torch.cuda.synchronize()
    assert int(status[0]) == moe.MOE_OK


def test_selftest_rejects_bad_arguments():
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    for polls in (0, (1 << 20) + 1):
        with pytest.raises(moe.MoeError):
            moe.selftest_bounded_wait(status, polls=polls)
