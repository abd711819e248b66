"""Device-side failure detection, exercised without faulting or hanging a GPU.

Every grouped-GEMM role waits through one bounded mbarrier wait that gives up
after a clock64 budget and records MOE_ERR_TIMEOUT in the status word of the
scratch buffer. moe_check_bounded_wait runs that wait on a barrier nothing
completes; the test checks that the status is reported, that clearing it works,
and that the context still runs a full layer correctly afterwards.
"""
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from workloads import TINY, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")


def test_bounded_wait_reports_timeout_and_context_survives():
    sz = B.moe_query_sizes(TINY)
    scratch = torch.zeros(int(sz.scratch_bytes), dtype=torch.uint8, device="cuda")
    assert B.moe_last_device_status(scratch) == 0
    B.moe_check_bounded_wait(scratch, 50_000_000)          # ~25 ms of SM clock
    assert B.moe_last_device_status(scratch) == 5          # MOE_ERR_TIMEOUT
    B.moe_clear_device_status(scratch)
    assert B.moe_last_device_status(scratch) == 0
    inp = make_inputs(TINY, seed=0)
    g = H_.run_layer(TINY, inp)                            # asserts status 0 itself
    H_.check_steps(TINY, inp, g)
