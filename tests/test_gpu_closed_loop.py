"""Receding-horizon pieces on the GPU against the oracle: the warm-start kernel (a pure data
move: bit-exact), the world-model simulator step, and the closed-loop episode, which must
equal the same steps driven one call at a time from the host (bitwise) and agree with
the oracle step by step, teacher-forced on the GPU's own states."""
import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from gpu_helpers import (TOL_BF16_ENERGY_REL, TOL_EPS, TOL_FP32_REL, cuda, host, make_planner,
                         oracle_weights_for, rel_err)
from oracle import cem, philox, predictor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [1, 2, 4])
def test_warm_start_matches_oracle_bitwise(H):
    p = make_planner("tiny", max_horizon=4)
    rng = np.random.default_rng(H)
    B = 3
    mu_prev = rng.uniform(-1, 1, (B, H, 7)).astype(np.float32)
    mu_pr = rng.standard_normal((B, H, 7)).astype(np.float32)
    sg_pr = rng.uniform(0.1, 2, (B, H, 7)).astype(np.float32)
    d_prev, d_mp, d_sp = cuda(mu_prev), cuda(mu_pr), cuda(sg_pr)
    mu_out, sg_out = torch.zeros(B, H, 7, device="cuda"), torch.zeros(B, H, 7, device="cuda")
    p.warm_start(d_prev, d_mp, d_sp, B, H, mu_out, sg_out)
    p.sync_check()
    for b in range(B):
        m_ref, s_ref = cem.warm_start(mu_prev[b], mu_pr[b], sg_pr[b])
        assert np.array_equal(host(mu_out)[b], m_ref.astype(np.float32))
        assert np.array_equal(host(sg_out)[b], s_ref.astype(np.float32))
    # in place: mu_out = mu_prev, sigma_out = sigma_prior
    p.warm_start(d_prev, d_mp, d_sp, B, H, d_prev, d_sp)
    p.sync_check()
    assert np.array_equal(host(d_prev), host(mu_out)) and np.array_equal(host(d_sp), sg_pr)
    p.close()


def _world_step(p, z, s, a, goal):
    B = z.shape[0]
    zn = torch.zeros_like(z)
    sn = torch.zeros_like(s)
    dist = torch.zeros(B, device="cuda")
    p.world_model_step(z, s, a, B, zn, sn, goal=goal, distance=dist)
    p.sync_check()
    return zn, sn, dist


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_world_model_step_matches_oracle(name):
    pc = {"tiny": synthetic.TINY, "small": synthetic.SMALL}[name]
    p = make_planner(name, max_horizon=1)
    B = 2
    z0, goal, s0 = synthetic.make_problems(pc, B)
    a = np.random.default_rng(5).uniform(-1, 1, (B, 7)).astype(np.float32)
    zn, sn, dist = _world_step(p, cuda(z0), cuda(s0), cuda(a), cuda(goal))
    w = oracle_weights_for(name)
    for b in range(B):
        z_ref, s_ref = cem.world_model_step(w, pc, z0[b], s0[b], a[b])
        d_ref = predictor.energy_l1(z_ref[None], goal[b])[0]
        if pc.precision == "fp32":
            assert np.max(np.abs(host(zn)[b] - z_ref)) / np.max(np.abs(z_ref)) < TOL_FP32_REL
            assert abs(host(dist)[b] - d_ref) / d_ref < TOL_FP32_REL
        else:
            assert np.linalg.norm(host(zn)[b] - z_ref) / np.linalg.norm(z_ref) < TOL_BF16_ENERGY_REL
            assert abs(host(dist)[b] - d_ref) / d_ref < TOL_BF16_ENERGY_REL
        assert np.array_equal(host(sn)[b], s0[b] + a[b])              # fp32 sum, same rounding
    # state_next may alias state
    s_d = cuda(s0)
    zn2 = torch.zeros_like(zn)
    p.world_model_step(cuda(z0), s_d, cuda(a), B, zn2, s_d)
    p.sync_check()
    assert np.array_equal(host(s_d), s0 + a) and torch.equal(zn2, zn)
    p.close()


def _episode(p, z0, s0, goal, mu_p, sg_p, H, N, K, R, steps, warm, seed):
    B = z0.shape[0]
    acts = torch.zeros(steps, B, 7, device="cuda")
    dist = torch.zeros(steps, B, device="cuda")
    p.closed_loop(cuda(z0), cuda(s0), cuda(goal), cuda(mu_p), cuda(sg_p), B, H, N, K, R, steps,
                  warm, seed, acts, dist)
    p.sync_check()
    return host(acts), host(dist)


def test_closed_loop_equals_host_driven_steps_and_oracle():
    wl = synthetic.WORKLOADS["tiny"]
    pc = wl.predictor
    H, N, K, R, steps, seed = 2, 64, 8, 2, 3, 17
    p = make_planner("tiny", max_horizon=H)
    B = 2
    z0, goal, s0 = synthetic.make_problems(pc, B)
    mu_p, sg_p = synthetic.make_gaussian(pc, B, H)
    acts, dist = _episode(p, z0, s0, goal, mu_p, sg_p, H, N, K, R, steps, 1, seed)

    # the same episode, one C-ABI call at a time, recording every intermediate state
    z, s = cuda(z0), cuda(s0)
    g = cuda(goal)
    mu0, sg0 = cuda(mu_p), cuda(sg_p)
    w = oracle_weights_for("tiny")
    for t in range(steps):
        a = torch.zeros(B, 7, device="cuda")
        tr = {"mu": torch.zeros(R + 1, B, H, 7, device="cuda"),
              "sigma": torch.zeros(R + 1, B, H, 7, device="cuda"),
              "actions": torch.zeros(R, B, N, H, 7, device="cuda"),
              "energy": torch.zeros(R, B, N, device="cuda")}
        p.plan(z, s, g, mu0, sg0, B, H, N, K, R, seed + t, a, trace=tr)
        zn, sn, d = _world_step(p, z, s, a, g)
        assert np.array_equal(host(a), acts[t]) and np.array_equal(host(d), dist[t])
        # oracle, teacher-forced on this step's GPU inputs
        trh = {k: host(v) for k, v in tr.items()}
        for b in range(B):
            eps = philox.sample_eps(seed + t, b, 0, N, H, 7)
            a_ref = philox.sample_actions(host(mu0)[b], host(sg0)[b], eps)
            assert np.max(np.abs(trh["actions"][0, b] - a_ref)) < TOL_EPS
            zb, sb = host(z)[b], host(s)[b]
            idx = [0, 7, N - 1]
            z_r = predictor.rollout(w, pc, zb, sb, trh["actions"][0, b][idx].astype(np.float64))[-1]
            assert rel_err(trh["energy"][0, b][idx], predictor.energy_l1(z_r, goal[b])) < TOL_FP32_REL
            z_ref, s_ref = cem.world_model_step(w, pc, zb, sb, host(a)[b])
            assert np.max(np.abs(host(zn)[b] - z_ref)) / np.max(np.abs(z_ref)) < TOL_FP32_REL
            assert abs(host(d)[b] - predictor.energy_l1(z_ref[None], goal[b])[0]) < \
                TOL_FP32_REL * host(d)[b]
        # next step's seed through the warm-start kernel, checked against the oracle's
        mu_n, sg_n = torch.zeros_like(mu0), torch.zeros_like(sg0)
        p.warm_start(tr["mu"][R], cuda(mu_p), cuda(sg_p), B, H, mu_n, sg_n)
        for b in range(B):
            m_next, s_next = cem.warm_start(trh["mu"][R, b], mu_p[b], sg_p[b])
            assert np.array_equal(host(mu_n)[b], m_next.astype(np.float32))
            assert np.array_equal(host(sg_n)[b], s_next.astype(np.float32))
        z, s, mu0, sg0 = zn, sn, mu_n, sg_n
    p.close()


def test_closed_loop_warm_start_is_a_no_op_at_horizon_one():
    pc = synthetic.TINY
    p = make_planner("tiny", max_horizon=1)
    z0, goal, s0 = synthetic.make_problems(pc, 1)
    mu_p, sg_p = synthetic.make_gaussian(pc, 1, 1)
    a0, d0 = _episode(p, z0, s0, goal, mu_p, sg_p, 1, 32, 4, 2, 3, 0, 5)
    a1, d1 = _episode(p, z0, s0, goal, mu_p, sg_p, 1, 32, 4, 2, 3, 1, 5)
    assert np.array_equal(a0, a1) and np.array_equal(d0, d1)
    from cem_search_transformer_gb300.binding import JepaError
    acts, dist = torch.zeros(1, 1, 7, device="cuda"), torch.zeros(1, 1, device="cuda")
    for steps, warm in ((0, 1), (1, 2)):
        with pytest.raises(JepaError) as ei:
            p.closed_loop(cuda(z0), cuda(s0), cuda(goal), cuda(mu_p), cuda(sg_p), 1, 1, 32, 4, 2,
                          steps, warm, 5, acts, dist)
        assert ei.value.status == 1
    p.close()
