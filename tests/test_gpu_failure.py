"""Failure detection on the GPU without a fault: every device wait is bounded.

A wait on something that nothing signals must end by itself, leave the
context usable and report MOE_ERR_TIMEOUT through the workspace error word.
"""
import time

import pytest
import torch

from combine_router_gemm_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1, 2], ids=["mbarrier", "lookback", "cluster_mbarrier"])
def test_bounded_wait_times_out_and_reports(which):
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    B.moe_selftest_bounded_wait(which, 20000, ws)  # 20 ms limit
    rc, detail = B.moe_check_error(ws)
    dt = time.perf_counter() - t0
    assert rc == B.ERR_TIMEOUT and detail != 0
    assert dt < 5.0
    # the context is still usable, and the error word was cleared by the check
    x = torch.ones(1000, device="cuda")
    assert float(x.sum()) == 1000.0
    rc, detail = B.moe_check_error(ws)
    assert rc == B.OK and detail == 0
