"""Shared setup for the GPU parity tests: seeded inputs, a loaded planner, tolerances."""
import functools

import numpy as np

from cem_search_transformer_gb300 import synthetic

# Tolerances (stated for the planning path): sampler Gaussians 1e-6 abs, integers exact;
# predictor 1e-4 rel in fp32 mode and 2e-2 rel per-candidate energy in bf16 mode;
# refit mean/std 1e-3.
TOL_EPS = 1e-6
TOL_FP32_REL = 1e-4
TOL_BF16_ENERGY_REL = 2e-2
TOL_REFIT = 1e-3


def cuda(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


@functools.lru_cache(maxsize=4)
def weights_for(name: str):
    return synthetic.make_weights(synthetic.PRESETS[name], seed=0)


@functools.lru_cache(maxsize=4)
def oracle_weights_for(name: str):
    from oracle import predictor
    return predictor.prepare_weights(weights_for(name), synthetic.PRESETS[name].precision)


def make_planner(name: str, max_horizon: int = 1, max_chunk: int = 0):
    from cem_search_transformer_gb300 import binding
    pc = synthetic.PRESETS[name]
    p = binding.Planner(pc, max_horizon=max_horizon, max_chunk=max_chunk)
    p.load_weights(weights_for(name))
    return p


def rel_err(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30))


def energy_gap_allows(energies_ref, K, tol_rel):
    """True when the K-th and (K+1)-th smallest reference energies differ by more than
    the tolerance, so any path within tolerance must pick the same elite set."""
    e = np.sort(np.asarray(energies_ref, np.float64))
    if K >= len(e):
        return True
    return (e[K] - e[K - 1]) > 2 * tol_rel * abs(e[K])
