"""Sampler row: Philox4x32-10 words bit-exact, Gaussians/actions within 1e-6 of the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL_EPS, cuda, host, make_planner
from oracle import philox

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def planner():
    p = make_planner("tiny", max_horizon=3)
    yield p
    p.close()


def test_philox_words_bit_exact(planner):
    rng = np.random.default_rng(0)
    n = 4099
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:4] = [[0, 0, 0, 0], [0xFFFFFFFF] * 4, [1, 2, 3, 4], [0, 0, 0, 0xFFFFFFFF]]
    for seed in (0, 42, 0xDEADBEEFCAFEF00D):
        out = torch.zeros(n, 4, dtype=torch.int32, device="cuda")
        planner.philox(cuda(ctr.view(np.int32)), seed, n, out)
        torch.cuda.synchronize()
        got = host(out).view(np.uint32)
        ref = np.stack(philox.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3],
                                            seed & 0xFFFFFFFF, seed >> 32), axis=1)
        assert np.array_equal(got, ref.astype(np.uint32))


@pytest.mark.parametrize("B,N,H,rnd", [(1, 800, 1, 0), (3, 37, 3, 5), (2, 1, 2, 9)])
def test_actions_match_oracle(planner, B, N, H, rnd):
    rng = np.random.default_rng(B * 100 + N)
    mu = rng.uniform(-0.5, 0.5, (B, H, 7)).astype(np.float32)
    sg = rng.uniform(0.05, 0.6, (B, H, 7)).astype(np.float32)
    seed = 1234567
    out = torch.zeros(B, N, H, 7, device="cuda")
    planner.sample_actions(cuda(mu), cuda(sg), B, N, H, rnd, seed, out)
    torch.cuda.synchronize()
    got = host(out)
    for b in range(B):
        eps = philox.sample_eps(seed, b, rnd, N, H, 7)
        ref = philox.sample_actions(mu[b], sg[b], eps)
        assert np.max(np.abs(got[b] - ref)) < TOL_EPS
        # recovered Gaussians where no clipping happened
        un = np.abs(ref) < 1.0 - 1e-6
        eps_got = (got[b].astype(np.float64) - mu[b][None]) / sg[b][None]
        assert np.max(np.abs(eps_got[un] - eps[un]) * sg[b][None].repeat(N, 0)[un]) < TOL_EPS


def test_unit_gaussian_draws(planner):
    """mu = 0, sigma = 1e-3 keeps everything unclipped: eps recovered to 1e-6 abs over 10^5 draws."""
    B, N, H = 1, 14336, 1
    mu = np.zeros((B, H, 7), np.float32)
    sg = np.full((B, H, 7), 1e-3, np.float32)
    out = torch.zeros(B, N, H, 7, device="cuda")
    planner.sample_actions(cuda(mu), cuda(sg), B, N, H, 3, 77, out)
    torch.cuda.synchronize()
    sigma = np.float64(np.float32(1e-3))
    eps_got = host(out)[0].astype(np.float64) / sigma
    eps = philox.sample_eps(77, 0, 3, N, H, 7)
    assert np.max(np.abs(eps_got - eps)) < TOL_EPS


def test_sigma_zero_and_clip(planner):
    mu = np.array([[[0.3, -2.0, 2.0, 0.0, 1.0, -1.0, 0.5]]], np.float32)
    out = torch.zeros(1, 5, 1, 7, device="cuda")
    planner.sample_actions(cuda(mu), cuda(np.zeros_like(mu)), 1, 5, 1, 0, 1, out)
    torch.cuda.synchronize()
    assert np.array_equal(host(out)[0, :, 0], np.broadcast_to(np.clip(mu[0, 0], -1, 1), (5, 7)))
