"""Candidates of one problem split across ranks (world sizes 2 and 3, gloo, 127.0.0.1, CPU).

Each rank draws all of a round's candidates, scores its own slice, and one all-gather of
the energies per round gives every rank the same input to the selection and refit. The
planner here is the oracle (one candidate rollout at a time, so that the energies are the
same bits however the candidates are sliced); the plan gathered this way equals the
single-process oracle plan bit for bit, as the planning page reports plans that do not
depend on the GPU count."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from cem_search_transformer_gb300 import sharded, synthetic
from oracle import cem, philox, predictor

PC = synthetic.TINY
N, K, R, H, SEED = 16, 4, 2, 2, 42


class OracleBackend:
    """The three steps of a sharded round computed by the oracle (torch CPU tensors)."""

    def __init__(self):
        self.w = predictor.prepare_weights(synthetic.make_weights(PC), PC.precision)

    def sample(self, mu, sigma, B, N_, H_, r, seed):
        return torch.from_numpy(np.stack([
            philox.sample_actions(mu[b].numpy(), sigma[b].numpy(),
                                  philox.sample_eps(seed, b, r, N_, H_, PC.action_dim))
            for b in range(B)]))

    def energies(self, z0, state0, goal, actions, H_):
        B, n = actions.shape[:2]
        out = np.zeros((B, n))
        for b in range(B):
            for i in range(n):
                z = predictor.rollout(self.w, PC, z0[b], state0[b], actions[b, i:i + 1].numpy())[-1]
                out[b, i] = predictor.energy_l1(z, goal[b])[0]
        return torch.from_numpy(out)

    def select_refit(self, energy, actions, K_):
        mus, sgs, els = [], [], []
        for b in range(actions.shape[0]):
            el = cem.select_elites(energy[b].numpy(), K_)
            m, s = cem.refit(actions[b].numpy()[el])
            mus.append(m), sgs.append(s), els.append(el)
        return torch.from_numpy(np.stack(mus)), torch.from_numpy(np.stack(sgs)), \
            torch.from_numpy(np.stack(els))

    @staticmethod
    def first_action(actions, winner):
        return actions[torch.arange(actions.shape[0]), winner.long(), 0]


def _inputs(B):
    z0, goal, s0 = synthetic.make_problems(PC, B)
    mu0, sg0 = synthetic.make_gaussian(PC, B, H)
    return z0, goal, s0, torch.from_numpy(mu0).double(), torch.from_numpy(sg0).double()


def _rank(rank, world, port, B, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    z0, goal, s0, mu0, sg0 = _inputs(B)
    action, trace = sharded.plan_sharded(OracleBackend(), z0, s0, goal, mu0, sg0, B, H, N, K, R,
                                         SEED, world, rank, sharded.torch_all_gather())
    tr = sharded.as_numpy_trace(trace)
    np.savez(f"{out_path}.{rank}.npz", action=action.numpy(), **tr)
    dist.destroy_process_group()


def _single_process_plan(b, z0, goal, s0):
    """The oracle's plan, one candidate rollout at a time (the same bits as any slicing)."""
    w = predictor.prepare_weights(synthetic.make_weights(PC), PC.precision)

    def energy_fn(actions):
        return np.array([predictor.energy_l1(
            predictor.rollout(w, PC, z0[b], s0[b], actions[i:i + 1])[-1], goal[b])[0]
            for i in range(actions.shape[0])])
    mu0, sg0 = synthetic.make_gaussian(PC, 1, H)
    return cem.cem_plan(energy_fn, mu0[0], sg0[0], N, K, R, SEED, b)


def test_slice_bounds_cover_candidates_once():
    for n in (1, 7, 16, 800, 801):
        for w in (1, 2, 3, 8):
            seen = np.concatenate([np.arange(*sharded.slice_bounds(n, w, r)) for r in range(w)])
            assert np.array_equal(seen, np.arange(n))
    with pytest.raises(ValueError):
        sharded.slice_bounds(10, 2, 2)


@pytest.mark.parametrize("world,B", [(2, 1), (3, 2)])
def test_sharded_candidates_reproduce_single_process_plan(tmp_path, world, B):
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        port = sck.getsockname()[1]
    out = str(tmp_path / "plan")
    mp.start_processes(_rank, args=(world, port, B, out), nprocs=world, join=True,
                       start_method="spawn")
    ranks = [np.load(f"{out}.{r}.npz") for r in range(world)]
    z0, goal, s0, _, _ = _inputs(B)
    for b in range(B):
        ref = _single_process_plan(b, z0, goal, s0)
        for got in ranks:              # every rank ends with the same plan
            assert np.array_equal(got["action"][b], ref["action"])
            assert np.array_equal(got["energy"][:, b], ref["energy"])
            assert np.array_equal(got["elites"][:, b], ref["elites"])
            assert np.array_equal(got["mu"][1:, b], ref["mu"][1:])
            assert np.array_equal(got["sigma"][1:, b], ref["sigma"][1:])
            assert got["winner"][b] == ref["winner"]
