"""Writes the oracle's energies for the full-shape bf16 parity tests with a reachable goal.

Calls only the oracle (``oracle/``) and the seeded generators: nothing here comes from the
CUDA path. For horizon H in (1, 3) of the full-shape predictor (24 x 1024, P = 256, E = 1408):

  * problem 0 of the synthetic recipe (z0, state0, and its independent N(0, 1) goal);
  * a hidden action sequence a* (``make_actions(seed=99)``); the reachable goal is the
    oracle's own last predicted frame for a*, so that candidate energies spread widely;
  * 800 candidates from ``make_actions(seed=23)``; 16 of them, evenly spaced, are rolled
    out by the oracle and scored against both goals.

Output: ``full_reachable_H{H}.json`` beside this script, with checksums of the inputs so
that a test can see that its regenerated inputs are the ones these energies belong to.

    python tests/golden/make_reachable_energies.py [H ...]
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from cem_search_transformer_gb300 import synthetic  # noqa: E402
from oracle import predictor  # noqa: E402

N_CAND = 800
SAMPLE = [int(i) for i in np.linspace(0, N_CAND - 1, 16).round()]
GOAL_SEED, CAND_SEED = 99, 23


def inputs(H):
    """Regenerates every input of the stored case (shared by the writer and the tests)."""
    pc = synthetic.FULL
    z0, goal_indep, s0 = synthetic.make_problems(pc, 1)
    astar = synthetic.make_actions(pc, 1, 1, H, seed=GOAL_SEED)[0]
    acts = synthetic.make_actions(pc, 1, N_CAND, H, seed=CAND_SEED)
    return pc, z0, goal_indep, s0, astar, acts


def reachable_goal(w, pc, z0, s0, astar):
    """The oracle's last predicted frame for the hidden sequence a* ([1, P, E] float32)."""
    return predictor.rollout(w, pc, z0[0], s0[0], astar.astype(np.float64))[-1][0][None].astype(np.float32)


def checksum(a):
    return float(np.asarray(a, np.float64).sum())


def main(hs):
    for H in hs:
        t0 = time.time()
        pc, z0, goal_indep, s0, astar, acts = inputs(H)
        w = predictor.prepare_weights(synthetic.make_weights(pc, seed=0), pc.precision)
        goal = reachable_goal(w, pc, z0, s0, astar)
        idx = np.array(SAMPLE)
        z = predictor.rollout(w, pc, z0[0], s0[0], acts[0][idx].astype(np.float64))[-1]
        rec = {"config": "full", "H": H, "n_candidates": N_CAND, "sample": SAMPLE,
               "goal_seed": GOAL_SEED, "candidate_seed": CAND_SEED,
               "checksum_z0": checksum(z0), "checksum_actions": checksum(acts),
               "checksum_reachable_goal": checksum(goal),
               "energy_reachable": predictor.energy_l1(z, goal[0]).tolist(),
               "energy_independent": predictor.energy_l1(z, goal_indep[0]).tolist(),
               "writer": "tests/golden/make_reachable_energies.py (oracle only)"}
        with open(os.path.join(HERE, f"full_reachable_H{H}.json"), "w") as f:
            json.dump(rec, f, indent=1)
        print(f"H={H}: {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main([int(a) for a in sys.argv[1:]] or [1, 3])
