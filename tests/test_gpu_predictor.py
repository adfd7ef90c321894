"""Predictor rows (embed, LN, QKV, block-causal attention with KV cache, out-proj, MLP,
out-projection + L1 energy) through jepa_predictor_forward, against the oracle."""
import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from gpu_helpers import (TOL_BF16_ENERGY_REL, TOL_FP32_REL, cuda, host, make_planner,
                         oracle_weights_for, rel_err)
from oracle import predictor

pytestmark = pytest.mark.gpu


def _inputs(pc, B, N, H, seed=3):
    z0, goal, s0 = synthetic.make_problems(pc, B, seed_base=2000 + seed)
    acts = synthetic.make_actions(pc, B, N, H, seed=seed)
    return z0, goal, s0, acts


def _run(planner, pc, z0, goal, s0, acts, want_z=True):
    B, N, H, _ = acts.shape
    E, P = pc.embed_dim, pc.patch_tokens
    zp = torch.zeros(B, N, P, E, device="cuda") if want_z else None
    en = torch.zeros(B, N, device="cuda")
    planner.predictor_forward(cuda(z0), cuda(s0), cuda(acts), B, N, H, goal=cuda(goal), z_pred=zp,
                              energy=en)
    planner.sync_check()
    return (host(zp) if want_z else None), host(en)


def _oracle(name, pc, z0, goal, s0, acts, b, idx):
    w = oracle_weights_for(name)
    z = predictor.rollout(w, pc, z0[b], s0[b], acts[b][idx].astype(np.float64))[-1]
    return z, predictor.energy_l1(z, goal[b])


@pytest.mark.parametrize("B,N,H", [(2, 37, 1), (1, 16, 3), (1, 1, 2)])
def test_tiny_fp32_matches_oracle(B, N, H):
    pc = synthetic.TINY
    p = make_planner("tiny", max_horizon=3)
    z0, goal, s0, acts = _inputs(pc, B, N, H)
    zp, en = _run(p, pc, z0, goal, s0, acts)
    for b in range(B):
        z_ref, e_ref = _oracle("tiny", pc, z0, goal, s0, acts, b, np.arange(N))
        assert np.max(np.abs(zp[b] - z_ref)) / np.max(np.abs(z_ref)) < TOL_FP32_REL
        assert rel_err(en[b], e_ref) < TOL_FP32_REL
    p.close()


@pytest.mark.parametrize("B,N,H", [(2, 24, 2), (1, 5, 1)])
def test_small_bf16_matches_oracle(B, N, H):
    pc = synthetic.SMALL
    p = make_planner("small", max_horizon=2)
    z0, goal, s0, acts = _inputs(pc, B, N, H)
    zp, en = _run(p, pc, z0, goal, s0, acts)
    for b in range(B):
        z_ref, e_ref = _oracle("small", pc, z0, goal, s0, acts, b, np.arange(N))
        assert rel_err(en[b], e_ref) < TOL_BF16_ENERGY_REL
        # the predicted frame itself: bf16 activations, fp32 accumulation
        assert np.max(np.abs(zp[b] - z_ref)) / np.max(np.abs(z_ref)) < 5e-2
        print(f"small bf16 b={b}: energy rel err {rel_err(en[b], e_ref):.2e}, "
              f"z rel err {np.max(np.abs(zp[b] - z_ref)) / np.max(np.abs(z_ref)):.2e}")
    p.close()


def test_chunk_permutation_and_batch_invariance():
    """Same candidates give bitwise-identical energies however they are chunked, ordered or
    batched with other problems (the planning page reports the same plans for GPU counts from one to eight)."""
    pc = synthetic.SMALL
    B, N, H = 2, 40, 2
    z0, goal, s0, acts = _inputs(pc, B, N, H, seed=5)
    p_full = make_planner("small", max_horizon=2)
    p_chunk = make_planner("small", max_horizon=2, max_chunk=7)
    _, e_full = _run(p_full, pc, z0, goal, s0, acts, want_z=False)
    _, e_chunk = _run(p_chunk, pc, z0, goal, s0, acts, want_z=False)
    assert np.array_equal(e_full, e_chunk)
    perm = np.random.default_rng(0).permutation(N)
    _, e_perm = _run(p_full, pc, z0, goal, s0, acts[:, perm].copy(), want_z=False)
    assert np.array_equal(e_perm, e_full[:, perm])
    for b in range(B):
        _, e_b = _run(p_full, pc, z0[b:b + 1], goal[b:b + 1], s0[b:b + 1], acts[b:b + 1], want_z=False)
        assert np.array_equal(e_b[0], e_full[b])
    p_full.close()
    p_chunk.close()


@pytest.mark.parametrize("H,N,sample", [(1, 800, (0, 411, 799)), (3, 800, (517,))])
def test_full_shape_sampled_candidates(H, N, sample):
    """Full-shape predictor (24 x 1024, 256 x 1408 latents) at N = 800 in one pass, the launch
    configuration of the planning benchmark; sampled candidates recomputed by the oracle."""
    pc = synthetic.FULL
    p = make_planner("full", max_horizon=H)
    z0, goal, s0 = synthetic.make_problems(pc, 1)
    acts = synthetic.make_actions(pc, 1, N, H, seed=11)
    en = torch.zeros(1, N, device="cuda")
    zp = torch.zeros(1, N, pc.patch_tokens, pc.embed_dim, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), 1, N, H, goal=cuda(goal), z_pred=zp, energy=en)
    p.sync_check()
    en = host(en)[0]
    idx = np.array(sample)
    z_ref, e_ref = _oracle("full", pc, z0, goal, s0, acts, 0, idx)
    assert rel_err(en[idx], e_ref) < TOL_BF16_ENERGY_REL
    zs = host(zp[0, torch.as_tensor(idx, device="cuda")])
    assert np.max(np.abs(zs - z_ref)) / np.max(np.abs(z_ref)) < 5e-2
    assert np.all(np.isfinite(en))
    print(f"full H={H}: energy rel err {rel_err(en[idx], e_ref):.2e}")
    p.close()


def test_forward_argument_errors():
    from cem_search_transformer_gb300.binding import JepaError
    p = make_planner("tiny", max_horizon=1)
    z = torch.zeros(1, 16, 64, device="cuda")
    s = torch.zeros(1, 7, device="cuda")
    a = torch.zeros(1, 2, 2, 7, device="cuda")
    e = torch.zeros(1, 2, device="cuda")
    with pytest.raises(JepaError) as ei:
        p.predictor_forward(z, s, a, 1, 2, 2, goal=z, energy=e)     # H > max_horizon
    assert ei.value.status == 2
    with pytest.raises(JepaError) as ei:
        p.predictor_forward(z, s, a, 1, 2, 1, energy=e)             # energy without goal
    assert ei.value.status == 1
    p.close()


@pytest.mark.parametrize("name,B,N,H", [("tiny_gated", 2, 37, 2), ("small_gated", 2, 24, 2)])
def test_gated_mlp_predictor_matches_oracle(name, B, N, H):
    """Gated-MLP variant (FC1 * GELU(FC2) up-projection, one GEMM over interleaved weights)
    through the whole predictor, fp32 (SIMT) and bf16 (tcgen05) paths, held to the same
    bounds as the GELU network."""
    pc = synthetic.PRESETS[name]
    p = make_planner(name, max_horizon=2)
    z0, goal, s0, acts = _inputs(pc, B, N, H, seed=7)
    zp, en = _run(p, pc, z0, goal, s0, acts)
    for b in range(B):
        z_ref, e_ref = _oracle(name, pc, z0, goal, s0, acts, b, np.arange(N))
        zerr = np.max(np.abs(zp[b] - z_ref)) / np.max(np.abs(z_ref))
        if pc.precision == "fp32":
            assert zerr < TOL_FP32_REL and rel_err(en[b], e_ref) < TOL_FP32_REL
        else:
            assert rel_err(en[b], e_ref) < TOL_BF16_ENERGY_REL and zerr < 5e-2
        print(f"{name} b={b}: energy rel err {rel_err(en[b], e_ref):.2e}, z rel err {zerr:.2e}")
    p.close()


def test_full_gated_sampled_candidates():
    """Full-shape gated predictor at N = 800 (the gated benchmark's launch configuration);
    sampled candidates recomputed by the oracle."""
    pc = synthetic.FULL_GATED
    p = make_planner("full_gated", max_horizon=1)
    z0, goal, s0 = synthetic.make_problems(pc, 1)
    acts = synthetic.make_actions(pc, 1, 800, 1, seed=12)
    en = torch.zeros(1, 800, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), 1, 800, 1, goal=cuda(goal), energy=en)
    p.sync_check()
    en = host(en)[0]
    idx = np.array([3, 640])
    _, e_ref = _oracle("full_gated", pc, z0, goal, s0, acts, 0, idx)
    assert rel_err(en[idx], e_ref) < TOL_BF16_ENERGY_REL and np.all(np.isfinite(en))
    print(f"full_gated: energy rel err {rel_err(en[idx], e_ref):.2e}")
    p.close()


@pytest.mark.parametrize("name,H", [("small", 2), ("tiny", 1), ("small_fp8", 1)])
def test_shared_frame0_rows_are_exact(name, H):
    """Frame 0's patch rows enter layer 0 identically for every candidate of a problem, so
    their LayerNorm and QKV product are computed once per problem (N > 1) and broadcast. A
    candidate scored alone (N = 1, every row computed per candidate) gets the same bits."""
    pc = synthetic.PRESETS[name]
    B, N = 2, 6
    z0, goal, s0, acts = _inputs(pc, B, N, H, seed=13)
    p = make_planner(name, max_horizon=H)
    zp, en = _run(p, pc, z0, goal, s0, acts)
    for b in range(B):
        for i in (0, N - 1):
            z1, e1 = _run(p, pc, z0[b:b + 1], goal[b:b + 1], s0[b:b + 1], acts[b:b + 1, i:i + 1].copy())
            assert np.array_equal(e1[0, 0], en[b, i]) and np.array_equal(z1[0, 0], zp[b, i])
    p.close()
