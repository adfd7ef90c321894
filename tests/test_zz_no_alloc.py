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
    # raw addresses skip the binding's size checks, so the library's own limit answers:
    # 2^20 candidates x 8 row blocks of 32 patches are beyond the fixed scratch, and the call
    # is refused before anything is launched
    with pytest.raises(binding.JepaError) as ei:
        binding.energy_l1_noalloc(z.data_ptr(), z.data_ptr(), 1 << 10, 1 << 10, 256, 4, z.data_ptr())
    assert ei.value.status == 2 and "fixed scratch" in str(ei.value)


def test_noalloc_energy_rejects_short_buffers():
    """Tensors too small for the stated shape are refused before the library is called."""
    B, N, P, E = 1, 3, 40, 64
    z = torch.zeros(B, N, P, E, device="cuda")
    g = torch.zeros(B, P, E, device="cuda")
    e = torch.zeros(B, N, device="cuda")
    for args in ((z, g[:, :-1], e), (z[:, :-1], g, e), (z, g, e[:, :-1]),
                 (z, g.to(torch.bfloat16), e), (z, g.transpose(1, 2), e)):
        with pytest.raises(binding.JepaError) as ei:
            binding.energy_l1_noalloc(args[0], args[1], B, N, P, E, args[2])
        assert ei.value.status == 1
