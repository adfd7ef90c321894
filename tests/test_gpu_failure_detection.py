"""Failure detection without a GPU fault: a bounded device-side wait that nothing completes
gives up after its limit, the kernel returns, the host reads JEPA_ERR_TIMEOUT, and the
context keeps working afterwards."""
import time

import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from cem_search_transformer_gb300.binding import JepaError
from gpu_helpers import cuda, host, make_planner

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_recovers():
    p = make_planner("tiny", max_horizon=1)
    t0 = time.time()
    p.selftest_bounded_wait()
    with pytest.raises(JepaError) as ei:
        p.sync_check()
    assert ei.value.status == 6                      # JEPA_ERR_TIMEOUT
    assert 1.5 < time.time() - t0 < 30.0             # the 2 s limit, not a hang
    p.sync_check()                                   # the flag was cleared
    # the context still plans normally
    z0, goal, s0 = synthetic.make_problems(synthetic.TINY, 1)
    mu0, sg0 = synthetic.make_gaussian(synthetic.TINY, 1, 1)
    out = torch.zeros(1, 7, device="cuda")
    p.plan(cuda(z0), cuda(s0), cuda(goal), cuda(mu0), cuda(sg0), 1, 1, 32, 4, 2, 3, out)
    p.sync_check()
    assert np.all(np.isfinite(host(out)))
    p.close()
