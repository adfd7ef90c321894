"""Cross-entropy-method planning loop: elites, Gaussian refit, rounds, winner.

Test infrastructure (see the package docstring). Follows "Real-time inference for
JEPA world-model architectures with Ray", section "Where the sixteen seconds
actually goes": in every round N action sequences are sampled from the current
Gaussian and given an energy, and the Gaussian is refitted to the K of lowest
energy; after R rounds the first action of the final round's lowest-energy
sequence is the output.

Readings taken where the page is silent:
  * "best" = lowest energy; ties go to the lower candidate index; NaN ranks last;
  * the refit is the elites' mean and population (maximum-likelihood) standard
    deviation per (horizon step, action dim), over the clipped actions that were
    scored; no smoothing, no variance floor;
  * the winner is the lowest-energy candidate of the final round and the returned
    action is its first step a[winner, 0, :].

Receding-horizon control (same page, section "Further Optimization", parts A and B):
the robot executes one action per planning step and the next step may be seeded from
the previous plan instead of a fresh Gaussian; that section's closed-loop experiments
let the predictor play the robot. Readings taken:
  * warm start: the last round's mean loses its executed first step, the remaining
    H-1 steps move one step earlier, and the newly exposed last step takes the prior's
    mean; every step's width restarts at the prior's sigma (re-using the mean, not the
    collapsed spread, so the search keeps exploring);
  * control step t plans with seed + t, so consecutive steps draw fresh candidates;
  * the simulator step feeds the executed action through the predictor with horizon 1
    (z_{t+1} = predicted frame, s_{t+1} = s_t + a_t) and the distance to the goal is
    the same L1 energy the planner minimises.
"""
from __future__ import annotations

from typing import Callable, Dict

import numpy as np

from . import philox, predictor


def select_elites(energy: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K lowest energies, ordered by (energy, index); NaN counts as +inf."""
    e = np.where(np.isnan(energy), np.inf, np.asarray(energy, np.float64))
    order = np.lexsort((np.arange(e.shape[0]), e))    # primary key e, then index
    return order[:K]


def refit(elite_actions: np.ndarray):
    """Mean and population std over the elite axis: [K, H, A] -> ([H, A], [H, A])."""
    a = np.asarray(elite_actions, np.float64)
    mu = a.mean(axis=0)
    sigma = np.sqrt(((a - mu[None]) ** 2).mean(axis=0))
    return mu, sigma


def cem_plan(energy_fn: Callable[[np.ndarray], np.ndarray], mu0: np.ndarray, sigma0: np.ndarray,
             N: int, K: int, rounds: int, seed: int, b: int = 0) -> Dict[str, np.ndarray]:
    """R rounds of CEM for one problem b with a caller-supplied energy.

    energy_fn maps actions [N, H, A] (float64) to energies [N].
    Returns the chosen first action and the per-round trace.
    """
    mu = np.asarray(mu0, np.float64)
    sigma = np.asarray(sigma0, np.float64)
    H, A = mu.shape
    trace = {"mu": [mu], "sigma": [sigma], "actions": [], "energy": [], "elites": []}
    for r in range(rounds):
        eps = philox.sample_eps(seed, b, r, N, H, A)
        a = philox.sample_actions(mu, sigma, eps)
        e = np.asarray(energy_fn(a), np.float64)
        elites = select_elites(e, K)
        mu, sigma = refit(a[elites])
        for key, val in (("actions", a), ("energy", e), ("elites", elites), ("mu", mu),
                         ("sigma", sigma)):
            trace[key].append(val)
    winner = int(trace["elites"][-1][0])
    out = {k: np.stack(v) for k, v in trace.items()}
    out["winner"] = winner
    out["action"] = trace["actions"][-1][winner, 0].copy()
    return out


def warm_start(mu_final: np.ndarray, mu_prior: np.ndarray, sigma_prior: np.ndarray):
    """Seed of the next planning step from the previous plan's last-round mean [H, A]:
    steps 1..H-1 move to 0..H-2, step H-1 and all widths come from the prior."""
    mu = np.array(mu_prior, np.float64, copy=True)
    mu[:-1] = np.asarray(mu_final, np.float64)[1:]
    sigma = np.array(sigma_prior, np.float64, copy=True)
    return mu, sigma


def closed_loop(plan_fn: Callable, step_fn: Callable, distance_fn: Callable, z0, s0,
                mu_prior: np.ndarray, sigma_prior: np.ndarray, steps: int,
                warm: bool) -> Dict[str, np.ndarray]:
    """Receding-horizon episode: plan, execute the first action, observe, replan.

    plan_fn(z, s, mu0, sigma0, t) -> (action [A], last-round mean [H, A]);
    step_fn(z, s, a) -> (z', s'); distance_fn(z') -> float.
    Returns per-step actions [steps, A], distances [steps] and the seeds' means
    [steps, H, A] (what each step started from).
    """
    z, s = z0, np.asarray(s0, np.float64)
    mu0, sg0 = np.asarray(mu_prior, np.float64), np.asarray(sigma_prior, np.float64)
    actions, dists, seeds = [], [], []
    for t in range(steps):
        seeds.append(mu0)
        a, mu_last = plan_fn(z, s, mu0, sg0, t)
        z, s = step_fn(z, s, np.asarray(a, np.float64))
        actions.append(np.asarray(a, np.float64))
        dists.append(float(distance_fn(z)))
        if warm:
            mu0, sg0 = warm_start(mu_last, mu_prior, sigma_prior)
    return {"actions": np.stack(actions), "distance": np.array(dists), "mu0": np.stack(seeds)}


def predictor_energy_fn(w: Dict[str, np.ndarray], cfg, z0: np.ndarray, state0: np.ndarray,
                        goal: np.ndarray) -> Callable[[np.ndarray], np.ndarray]:
    """Energy of each candidate: L1 distance of its final predicted frame to the goal."""
    def fn(actions: np.ndarray) -> np.ndarray:
        preds = predictor.rollout(w, cfg, z0, state0, actions)
        return predictor.energy_l1(preds[-1], goal)
    return fn


def plan(weights_fp32: Dict[str, np.ndarray], cfg, z0: np.ndarray, state0: np.ndarray,
         goal: np.ndarray, mu0: np.ndarray, sigma0: np.ndarray, N: int, K: int, rounds: int,
         seed: int, b: int = 0) -> Dict[str, np.ndarray]:
    """Full planning step for problem b (z0, goal [P, E]; state0 [S]; mu0, sigma0 [H, A])."""
    w = predictor.prepare_weights(weights_fp32, cfg.precision)
    return cem_plan(predictor_energy_fn(w, cfg, z0, state0, goal), mu0, sigma0, N, K, rounds,
                    seed, b)


def world_model_step(w: Dict[str, np.ndarray], cfg, z: np.ndarray, s: np.ndarray, a: np.ndarray):
    """Simulator step with the predictor standing in for the robot: z [P, E], s [S], a [A]."""
    a = np.asarray(a, np.float64)
    z_next = predictor.rollout(w, cfg, z, s, a[None, None, :])[-1][0]
    return z_next, np.asarray(s, np.float64) + a


def predictor_closed_loop(weights_fp32: Dict[str, np.ndarray], cfg, z0: np.ndarray,
                          state0: np.ndarray, goal: np.ndarray, mu_prior: np.ndarray,
                          sigma_prior: np.ndarray, N: int, K: int, rounds: int, seed: int,
                          steps: int, warm: bool, b: int = 0) -> Dict[str, np.ndarray]:
    """Closed-loop episode of problem b, planning and simulating with the same predictor."""
    w = predictor.prepare_weights(weights_fp32, cfg.precision)

    def plan_fn(z, s, mu0, sg0, t):
        out = cem_plan(predictor_energy_fn(w, cfg, z, s, goal), mu0, sg0, N, K, rounds,
                       seed + t, b)
        return out["action"], out["mu"][-1]

    return closed_loop(plan_fn, lambda z, s, a: world_model_step(w, cfg, z, s, a),
                       lambda z: predictor.energy_l1(z[None], goal)[0], z0, state0, mu_prior,
                       sigma_prior, steps, warm)
