"""The allocation-free energy entry point (for callers that cannot allocate device memory,
such as a process under a fixed memory budget owned by a host framework, or a control loop
that must not allocate mid-episode) agrees with the energies jepa_predictor_forward computes
through its regular workspace, on two calls in a row.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import binding, synthetic
from gpu_helpers import TOL_FP32_REL, cuda, host, make_planner, rel_err

pytestmark = pytest.mark.gpu


def test_noalloc_energy_matches_predictor_forward():
    pc = synthetic.SMALL
    B, N, H = 2, 24, 2
    P, E = pc.patch_tokens, pc.embed_dim
    z0, goal, s0 = synthetic.make_problems(pc, B, seed_base=3000)
    acts = synthetic.make_actions(pc, B, N, H, seed=21)
    p = make_planner("small", max_horizon=H)
    z_pred = torch.zeros(B, N, P, E, device="cuda")
    e_ref = torch.zeros(B, N, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), B, N, H, goal=cuda(goal), z_pred=z_pred,
                        energy=e_ref)
    p.sync_check()
    g = cuda(goal)
    # first call: every problem and candidate
    e1 = torch.full((B, N), -1.0, device="cuda")
    binding.energy_l1_noalloc(z_pred, g, B, N, P, E, e1)
    torch.cuda.synchronize()
    assert rel_err(host(e1), host(e_ref)) < TOL_FP32_REL
    # second call right after, on a different (smaller) slice: the shared scratch still
    # holds the first call's partial sums, which must not leak into this result
    e2 = torch.full((1, N - 5), -1.0, device="cuda")
    binding.energy_l1_noalloc(z_pred[1:, 5:].contiguous(), g[1:].contiguous(), 1, N - 5, P, E, e2)
    torch.cuda.synchronize()
    assert rel_err(host(e2)[0], host(e_ref)[1, 5:]) < TOL_FP32_REL
    p.close()


def test_noalloc_energy_rejects_oversized_batches():
    z = torch.zeros(1, 4, device="cuda")
    with pytest.raises(binding.JepaError) as ei:
        # 2^20 candidates x 8 row blocks of 32 patches: beyond the fixed scratch
        binding.energy_l1_noalloc(z, z, 1 << 10, 1 << 10, 256, 4, z)
    assert ei.value.status == 2 and "fixed scratch" in str(ei.value)
