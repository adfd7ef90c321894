"""Candidate sharding through the C ABI on one GPU: the rank logic of sharded.plan_sharded
driven by the library's entry points equals the captured-graph plan (jepa_cem_plan) bit for
bit. World size 1 is the real path; world sizes 2 and 3 run each rank as a host thread with
its own context, exchanging energies through host memory after a device synchronisation
(no kernel of one rank waits on another's)."""
import threading

import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import sharded, synthetic
from gpu_helpers import cuda, host, make_planner

pytestmark = pytest.mark.gpu


def _graph_plan(wl, z0, goal, s0, mu0, sg0):
    B, N, K, R, H = z0.shape[0], wl.N, wl.K, wl.rounds, wl.horizon
    p = make_planner(wl.predictor.name, max_horizon=H)
    out = torch.zeros(B, 7, device="cuda")
    tr = {"mu": torch.zeros(R + 1, B, H, 7, device="cuda"),
          "sigma": torch.zeros(R + 1, B, H, 7, device="cuda"),
          "energy": torch.zeros(R, B, N, device="cuda"),
          "elites": torch.zeros(R, B, K, dtype=torch.int32, device="cuda"),
          "winner": torch.zeros(B, dtype=torch.int32, device="cuda")}
    p.plan(cuda(z0), cuda(s0), cuda(goal), cuda(mu0), cuda(sg0), B, H, N, K, R, wl.seed, out, trace=tr)
    p.sync_check()
    p.close()
    return host(out), {k: host(v) for k, v in tr.items()}


class _HostGather:
    """all_gather among host threads: each deposits its buffer, waits for the others."""

    def __init__(self, world):
        self.world = world
        self.slots = [None] * world
        self.barrier = threading.Barrier(world, timeout=120)

    def for_rank(self, rank):
        def fn(buf):
            torch.cuda.synchronize()
            self.slots[rank] = buf.clone()
            torch.cuda.synchronize()
            self.barrier.wait()
            parts = list(self.slots)
            self.barrier.wait()
            return parts
        return fn


@pytest.mark.parametrize("world,B", [(1, 1), (2, 1), (3, 2)])
def test_sharded_plan_equals_graph_plan(world, B):
    wl = synthetic.WORKLOADS["small"]
    pc, N, K, R, H = wl.predictor, wl.N, wl.K, wl.rounds, wl.horizon
    z0, goal, s0 = synthetic.make_problems(pc, B)
    mu0, sg0 = synthetic.make_gaussian(pc, B, H)
    ref_out, ref = _graph_plan(wl, z0, goal, s0, mu0, sg0)
    gather = _HostGather(world)
    results, errors = [None] * world, []

    def run(rank):
        try:
            p = make_planner(pc.name, max_horizon=H)
            action, trace = sharded.plan_sharded(
                sharded.CudaBackend(p), cuda(z0), cuda(s0), cuda(goal), cuda(mu0), cuda(sg0), B, H,
                N, K, R, wl.seed, world, rank, gather.for_rank(rank))
            p.sync_check()
            results[rank] = (host(action), sharded.as_numpy_trace(trace))
            p.close()
        except Exception as e:          # reported on the main thread
            errors.append(e)
            gather.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for action, tr in results:
        assert np.array_equal(action, ref_out)
        assert np.array_equal(tr["energy"], ref["energy"])
        assert np.array_equal(tr["elites"], ref["elites"])
        assert np.array_equal(tr["mu"], ref["mu"])
        assert np.array_equal(tr["sigma"], ref["sigma"])
        assert np.array_equal(tr["winner"], ref["winner"])
