"""Cross-entropy-method planning loop: elites, Gaussian refit, rounds, winner.

Test infrastructure (see the package docstring). Follows "Real-time inference for
JEPA world-model architectures with Ray", section "Where the sixteen seconds
actually goes": each round draws N candidate action sequences from a Gaussian
centred on the current guess, scores every one, keeps the best K and re-centres
the Gaussian on them; after R rounds only the first action of the winning
sequence is executed.

Readings taken where the page is silent:
  * "best" = lowest energy; ties go to the lower candidate index; NaN ranks last;
  * the refit is the elites' mean and population (maximum-likelihood) standard
    deviation per (horizon step, action dim), over the clipped actions that were
    scored; no smoothing, no variance floor;
  * the winner is the lowest-energy candidate of the final round and the returned
    action is its first step a[winner, 0, :].
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
