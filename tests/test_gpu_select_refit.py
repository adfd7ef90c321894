"""Elite selection + refit row: elites bit-exact vs the oracle on the same energies, refit within 1e-3."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL_REFIT, cuda, host, make_planner
from oracle import cem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def planner():
    p = make_planner("tiny", max_horizon=3)
    yield p
    p.close()


@pytest.mark.parametrize("B,N,K,H,ties", [(1, 800, 80, 1, False), (3, 200, 20, 2, True),
                                          (2, 1, 1, 1, False), (1, 3200, 320, 1, True),
                                          (1, 8192, 819, 1, False), (2, 100, 100, 3, True)])
def test_select_refit_matches_oracle(planner, B, N, K, H, ties):
    rng = np.random.default_rng(N + K)
    e = rng.standard_normal((B, N)).astype(np.float32)
    if ties:
        e = np.round(e * 4) / 4          # many exact ties, including -0.0 against +0.0
        e[:, ::17] = np.nan
    a = rng.uniform(-1, 1, (B, N, H, 7)).astype(np.float32)
    mu = torch.zeros(B, H, 7, device="cuda")
    sg = torch.zeros(B, H, 7, device="cuda")
    el = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    planner.select_refit(cuda(e), cuda(a), B, N, H, K, mu, sg, el)
    torch.cuda.synchronize()
    for b in range(B):
        ref_el = cem.select_elites(e[b], K)
        assert np.array_equal(host(el)[b], ref_el)
        m_ref, s_ref = cem.refit(a[b][ref_el])
        assert np.max(np.abs(host(mu)[b] - m_ref)) < TOL_REFIT * 1e-2
        assert np.max(np.abs(host(sg)[b] - s_ref)) < TOL_REFIT * 1e-2


def test_select_rejects_bad_k(planner):
    from cem_search_transformer_gb300.binding import JepaError
    z = torch.zeros(1, 4, device="cuda")
    a = torch.zeros(1, 4, 1, 7, device="cuda")
    m = torch.zeros(1, 1, 7, device="cuda")
    with pytest.raises(JepaError) as ei:
        planner.select_refit(z, a, 1, 4, 1, 5, m, m)
    assert ei.value.status == 1
