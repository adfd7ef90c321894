"""Pins for the oracle's CEM loop: brute-force top-K, closed-form refit, special cases and
convergence to the closed-form optimum of a linear-quadratic problem (CPU only)."""
import numpy as np

from oracle import cem, philox


def test_select_elites_brute_force():
    rng = np.random.default_rng(0)
    for trial in range(50):
        n = int(rng.integers(1, 60))
        e = rng.integers(0, 6, n).astype(np.float64) * 0.5     # many ties
        e[rng.random(n) < 0.1] = np.nan
        k = int(rng.integers(1, n + 1))
        key = lambda i: (np.inf if np.isnan(e[i]) else e[i], i)
        want = sorted(range(n), key=key)[:k]
        assert list(cem.select_elites(e, k)) == want


def test_refit_closed_form():
    a = np.array([[[1.0, -1.0]], [[3.0, -1.0]], [[5.0, -1.0]], [[7.0, -1.0]]])   # [K=4, H=1, A=2]
    mu, sigma = cem.refit(a)
    assert np.allclose(mu, [[4.0, -1.0]]) and np.allclose(sigma, [[np.sqrt(5.0), 0.0]])


def test_sigma_zero_gives_identical_candidates():
    calls = []
    def energy(a):
        calls.append(a)
        return np.abs(a).sum(axis=(1, 2))
    mu0 = np.full((2, 7), 0.3)
    out = cem.cem_plan(energy, mu0, np.zeros((2, 7)), N=16, K=4, rounds=2, seed=5)
    assert np.all(calls[0] == 0.3)
    assert list(out["elites"][0]) == [0, 1, 2, 3]
    assert np.allclose(out["sigma"][1], 0) and np.allclose(out["mu"][1], 0.3)
    assert out["winner"] == 0 and np.allclose(out["action"], 0.3)


def test_k_equals_n_refits_sample_moments():
    out = cem.cem_plan(lambda a: a.sum(axis=(1, 2)), np.zeros((1, 7)), np.ones((1, 7)),
                       N=50, K=50, rounds=1, seed=9)
    a = out["actions"][0]
    assert np.allclose(out["mu"][1], a.mean(0)) and np.allclose(out["sigma"][1], a.std(0))


def test_trace_consistency():
    out = cem.cem_plan(lambda a: (a ** 2).sum(axis=(1, 2)), np.zeros((2, 7)), np.ones((2, 7)),
                       N=40, K=5, rounds=3, seed=11, b=2)
    for r in range(3):
        eps = philox.sample_eps(11, 2, r, 40, 2, 7)
        a = philox.sample_actions(out["mu"][r], out["sigma"][r], eps)
        assert np.array_equal(a, out["actions"][r])
        assert out["energy"][r][out["elites"][r][0]] == out["energy"][r].min()
    assert np.array_equal(out["action"], out["actions"][2][out["winner"], 0])


def test_cem_converges_to_linear_quadratic_optimum():
    """Linear predictor z(a) = z0 + M vec(a), energy |z(a) - g|^2: the optimum is the
    least-squares solution (M^T M)^-1 M^T (g - z0), placed inside the action box."""
    rng = np.random.default_rng(3)
    H, A, D = 2, 7, 30
    M = rng.standard_normal((D, H * A))
    a_star = rng.uniform(-0.6, 0.6, H * A)
    z0 = rng.standard_normal(D)
    g = z0 + M @ a_star + 0.05 * rng.standard_normal(D)          # slightly off the range of M
    ls = np.linalg.solve(M.T @ M, M.T @ (g - z0))
    assert np.all(np.abs(ls) < 0.9)
    energy = lambda a: ((z0[None] + a.reshape(len(a), -1) @ M.T - g[None]) ** 2).sum(1)
    # the planning page's search (800 x keep 80 x 10 rounds) gets close; more rounds get closer
    out10 = cem.cem_plan(energy, np.zeros((H, A)), np.ones((H, A)), N=800, K=80, rounds=10, seed=42)
    assert np.max(np.abs(out10["mu"][-1].ravel() - ls)) < 5e-2
    out = cem.cem_plan(energy, np.zeros((H, A)), np.ones((H, A)), N=800, K=80, rounds=20, seed=42)
    assert np.max(np.abs(out["mu"][-1].ravel() - ls)) < 1e-2
    assert np.max(np.abs(out["action"] - ls[:A])) < 1e-2
    assert np.all(out["sigma"][-1] < out["sigma"][0])
