"""Pins for the oracle's receding-horizon pieces (warm start, closed-loop episode) against
closed forms of a linear system with an endpoint energy (CPU only).

The system is x_{t+1} = x_t + a_t with energy |x_H - g|^2 of an H-step plan, so a plan's
energy depends only on the sum of its actions. That gives two exact facts:
  * after executing the first action of a plan, the warm-started mean (steps moved one
    earlier, prior mean 0 appended) reaches the same endpoint, hence the same energy;
  * with a planner that returns the minimum-norm exact plan (every step (g - x) / H),
    the closed-loop distance shrinks by the factor (1 - 1/H) per step.
A shift in the wrong direction, a wrong fill value or an off-by-one in the episode's
bookkeeping breaks one of them.
"""
import numpy as np

from oracle import cem


def _endpoint_energy(x, g, plan):
    return float(np.sum((x + plan.sum(axis=0) - g) ** 2))


def test_warm_start_horizon_one_is_the_prior():
    rng = np.random.default_rng(0)
    mu_final = rng.uniform(-1, 1, (1, 7))
    mu_p, sg_p = rng.standard_normal((1, 7)), rng.uniform(0.5, 2, (1, 7))
    mu, sg = cem.warm_start(mu_final, mu_p, sg_p)
    assert np.array_equal(mu, mu_p) and np.array_equal(sg, sg_p)


def test_warm_start_keeps_the_endpoint_of_the_executed_plan():
    rng = np.random.default_rng(1)
    for H in (2, 3, 5):
        x, g = rng.standard_normal(7), rng.standard_normal(7)
        mu_final = rng.uniform(-0.5, 0.5, (H, 7))
        before = _endpoint_energy(x, g, mu_final)
        mu_w, sg_w = cem.warm_start(mu_final, np.zeros((H, 7)), np.ones((H, 7)))
        after = _endpoint_energy(x + mu_final[0], g, mu_w)
        assert abs(after - before) < 1e-12 * max(1.0, before)
        assert np.array_equal(sg_w, np.ones((H, 7)))
        # a non-zero prior mean lands exactly in the new last step
        mu_w2, _ = cem.warm_start(mu_final, np.full((H, 7), 0.25), np.ones((H, 7)))
        assert np.array_equal(mu_w2[-1], np.full(7, 0.25))
        assert np.array_equal(mu_w2[:-1], mu_final[1:])


def test_closed_loop_with_exact_planner_closed_form():
    H, steps = 4, 6
    rng = np.random.default_rng(2)
    x0, g = rng.standard_normal(7) * 0.3, rng.standard_normal(7) * 0.3

    def plan_fn(z, s, mu0, sg0, t):
        plan = np.repeat(((g - s) / H)[None], H, axis=0)
        return plan[0], plan

    out = cem.closed_loop(plan_fn, lambda z, s, a: (z, s + a),
                          lambda z: 0.0, None, x0, np.zeros((H, 7)), np.ones((H, 7)), steps,
                          warm=True)
    x = x0.copy()
    for t in range(steps):
        want = (g - x0) / H * (1 - 1 / H) ** t
        assert np.allclose(out["actions"][t], want, atol=1e-14)
        x = x + out["actions"][t]
    assert np.allclose(g - x, (g - x0) * (1 - 1 / H) ** steps, atol=1e-14)
    # the seed of step t >= 1 is the previous plan shifted, prior mean 0 at the end
    for t in range(1, steps):
        prev = (g - x0) / H * (1 - 1 / H) ** (t - 1)
        assert np.allclose(out["mu0"][t][:-1], np.repeat(prev[None], H - 1, 0), atol=1e-14)
        assert np.array_equal(out["mu0"][t][-1], np.zeros(7))


def test_cem_closed_loop_on_linear_system_reaches_the_goal():
    """CEM as the planner on the same system with a running cost sum_h |x_h - g|^2 (so the
    first action matters): fresh and warm-started episodes both close the distance, and
    10 rounds per step end nearer the goal than 3 (plan quality vs rounds)."""
    H, steps, N, K = 3, 6, 200, 20
    rng = np.random.default_rng(4)
    x0, g = np.zeros(7), rng.uniform(-0.8, 0.8, 7)

    def make_plan(rounds):
        def plan_fn(z, s, mu0, sg0, t):
            e = lambda a: ((s[None, None] + np.cumsum(a, axis=1) - g[None, None]) ** 2).sum(
                axis=(1, 2))
            out = cem.cem_plan(e, mu0, sg0, N, K, rounds, 100 + t)
            return out["action"], out["mu"][-1]
        return plan_fn

    d0 = np.sum((x0 - g) ** 2)
    tail = {}
    for rounds in (3, 10):
        for warm in (False, True):
            out = cem.closed_loop(make_plan(rounds), lambda z, s, a: (z, s + a),
                                  lambda z: 0.0, None, x0, np.zeros((H, 7)), np.ones((H, 7)),
                                  steps, warm)
            xs = x0 + np.cumsum(out["actions"], axis=0)
            tail[(rounds, warm)] = np.mean(np.sum((xs[-3:] - g) ** 2, axis=1))
            assert tail[(rounds, warm)] < 0.8 * d0
    for warm in (False, True):
        assert tail[(10, warm)] < 0.1 * d0
        assert tail[(10, warm)] < tail[(3, warm)]
