"""Failure detection without a GPU fault: the library's on-chip waits are
bounded.  A self-test kernel waits, with the same helper as the data-path
kernels, on a barrier that nothing completes; the wait must give up after
about a second, report EP_STATUS_TIMEOUT through the status word, and leave
the context usable for the next calls."""
import time

import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_inputs
from gpu_util import assert_rows_equal, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ep.ep_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == ep.EP_STATUS_TIMEOUT
    assert 0.5 < elapsed < 30.0
    # the context still works: a full step on the tiny workload, against the oracle
    inp = make_inputs("tiny", seed=3)
    cfg = inp["cfg"]
    dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W)
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).cuda()
    out = dc.step(x, torch.from_numpy(inp["topk_idx"]).cuda(), torch.from_numpy(inp["topk_w"]).cuda())
    torch.cuda.synchronize()
    want = oracle.run_all(inp)["combine"]["out"]
    assert_rows_equal(u16(out), want, "out")
    assert int(dc.status.item()) == 0
