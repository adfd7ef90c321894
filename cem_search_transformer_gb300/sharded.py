"""One planning problem's candidates split across ranks (one process per GPU).

"Real-time inference for JEPA world-model architectures with Ray", section "02 · The
Approach": the rollouts of one round do not depend on each other, so they can be computed
on different GPUs and gathered before the round moves on; section "Measured on 8x A100"
reports the same plan for a given seed at every GPU count. Here, per round r:

  1. every rank draws all N candidates of the round itself. The sampler's Philox counters
     depend only on (seed, problem, candidate, round, step, dim), so no actions are sent
     and every rank holds the same bits;
  2. rank w rolls out and scores its slice n in [w N / W, (w + 1) N / W) of every problem;
  3. one all-gather puts the B x N energies (fp32) on every rank;
  4. every rank runs the same elite selection and refit on the same energies and actions,
     so the Gaussians, and the plan, stay identical across ranks with no further exchange.

After R rounds every rank holds the winner (the final round's lowest energy) and its first
action. The energies of a slice are bitwise those of the same candidates in a one-rank pass
(the predictor's results do not depend on how candidates are chunked), so the plan does not
depend on W.

The steps run through a backend with three calls, so the rank logic is the same whatever
computes them: ``CudaBackend`` drives the C-ABI library (each call one of its entry points,
the gather an NCCL all-gather through torch.distributed). No kernel reads another GPU's
memory.
"""
from __future__ import annotations

from typing import Callable, Tuple

import numpy as np


def slice_bounds(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Candidates [lo, hi) of rank `rank` out of `world` (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return rank * N // world, (rank + 1) * N // world


def gather_energies(local, N: int, world: int, rank: int, all_gather: Callable):
    """[B, N] energies from every rank's [B, hi - lo] slice, in candidate order.

    `all_gather(buf)` receives this rank's [B, S] buffer (S = the largest slice, padded) and
    returns the list of all ranks' buffers, rank order."""
    import torch
    B = local.shape[0]
    S = -(-N // world)
    buf = torch.zeros(B, S, dtype=local.dtype, device=local.device)
    buf[:, :local.shape[1]] = local
    parts = all_gather(buf)
    out = torch.empty(B, N, dtype=local.dtype, device=local.device)
    for w, part in enumerate(parts):
        lo, hi = slice_bounds(N, world, w)
        out[:, lo:hi] = part[:, :hi - lo]
    return out


def torch_all_gather(group=None):
    """all_gather over torch.distributed (NCCL for CUDA tensors, gloo for host tensors)."""
    import torch.distributed as dist

    def fn(buf):
        parts = [buf.new_empty(buf.shape) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, buf.contiguous(), group=group)
        return parts
    return fn


def plan_sharded(backend, z0, state0, goal, mu0, sigma0, B: int, H: int, N: int, K: int,
                 rounds: int, seed: int, world: int, rank: int, all_gather: Callable):
    """One planning step with the candidates of every round split over `world` ranks.

    backend.sample(mu, sigma, B, N, H, r, seed)            -> actions [B, N, H, A]
    backend.energies(z0, state0, goal, actions_slice, H)   -> energies [B, n] of the slice
    backend.select_refit(energies, actions, K)             -> (mu', sigma', elites [B, K])
    Returns (action [B, A], trace dict of mu, sigma, energy, elites per round, winner)."""
    if not (1 <= K <= N) or rounds < 1 or H < 1 or B < 1:
        raise ValueError("plan_sharded: need B, H, rounds >= 1 and 1 <= K <= N")
    lo, hi = slice_bounds(N, world, rank)
    mu, sigma = mu0, sigma0
    trace = {"mu": [mu0], "sigma": [sigma0], "energy": [], "elites": []}
    actions = None
    for r in range(rounds):
        actions = backend.sample(mu, sigma, B, N, H, r, seed)
        local = backend.energies(z0, state0, goal, actions[:, lo:hi], H)
        energy = gather_energies(local, N, world, rank, all_gather)
        mu, sigma, elites = backend.select_refit(energy, actions, K)
        for k, v in (("mu", mu), ("sigma", sigma), ("energy", energy), ("elites", elites)):
            trace[k].append(v)
    winner = trace["elites"][-1][:, 0]
    action = backend.first_action(actions, winner)
    trace["winner"] = winner
    return action, trace


class CudaBackend:
    """The three steps through the C-ABI library on this rank's GPU (torch CUDA tensors)."""

    def __init__(self, planner, stream=None):
        self.p = planner
        self.stream = stream

    def sample(self, mu, sigma, B, N, H, r, seed):
        import torch
        out = torch.empty(B, N, H, self.p.pc.action_dim, device=mu.device)
        self.p.sample_actions(mu, sigma, B, N, H, r, seed, out, stream=self.stream)
        return out

    def energies(self, z0, state0, goal, actions, H):
        import torch
        B, n = actions.shape[:2]
        out = torch.empty(B, n, device=actions.device)
        if n:
            self.p.predictor_forward(z0, state0, actions.contiguous(), B, n, H, goal=goal, energy=out,
                                     stream=self.stream)
        return out

    def select_refit(self, energy, actions, K):
        import torch
        B, N, H, A = actions.shape
        mu = torch.empty(B, H, A, device=actions.device)
        sigma = torch.empty(B, H, A, device=actions.device)
        elites = torch.empty(B, K, dtype=torch.int32, device=actions.device)
        self.p.select_refit(energy.contiguous(), actions, B, N, H, K, mu, sigma, elites,
                            stream=self.stream)
        return mu, sigma, elites

    @staticmethod
    def first_action(actions, winner):
        import torch
        b = torch.arange(actions.shape[0], device=actions.device)
        return actions[b, winner.long(), 0]


def as_numpy_trace(trace):
    """Trace lists stacked into arrays on the host (for comparisons)."""
    out = {}
    for k, v in trace.items():
        if isinstance(v, list):
            out[k] = np.stack([np.asarray(x.cpu() if hasattr(x, "cpu") else x) for x in v])
        else:
            out[k] = np.asarray(v.cpu() if hasattr(v, "cpu") else v)
    return out
