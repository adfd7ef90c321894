"""Seeded synthetic inputs for the CEM planning path.

This module only draws random numbers and fixes shapes. It holds none of the
method's arithmetic, so both the CUDA path (tests, bench) and the CPU oracle can
take their inputs from it without sharing any computation.

Workload shapes follow the V-JEPA2-AC planning walk-through ("Real-time inference
for JEPA world-model architectures with Ray", section "Where the sixteen seconds
actually goes": 800 candidates, keep 80, 10 rounds) with the predictor shapes of
the five synthetic configurations: tiny (fp32), small (bf16, horizon 2),
full-shape (24 x 1024, 256 x 1408 latents), multi-step (horizon 3) and the
throughput sweep.

Recipe (all numpy ``default_rng``, platform independent):
  * weights: seed 0; linear weights, biases, embeddings and positions ~ N(0, 0.02);
    LayerNorm gain 1 + N(0, 0.02), shift N(0, 0.02);
  * problem b: z0, goal ~ N(0, 1) of shape [P, E] from seed 1000 + b;
    state0 = 0.1 * N(0, 1) of shape [S] from the same stream;
  * CEM: mu0 = 0, sigma0 = 1, seed 42.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np


@dataclasses.dataclass(frozen=True)
class PredictorConfig:
    """Shape of the action-conditioned predictor and of one planning problem."""

    name: str
    layers: int
    width: int          # d
    heads: int          # h
    mlp: int            # m
    patch_tokens: int   # P
    embed_dim: int      # E
    action_dim: int = 7  # A
    state_dim: int = 7   # S
    precision: str = "bf16"  # "fp32", "bf16" or "fp8" (bf16 with fp8 LayerNorm-fed GEMMs)
    ln_eps: float = 1e-5
    mlp_kind: str = "gelu"   # "gelu": W_2 GELU(W_1 x); "gated": W_2 (W_1 x * GELU(W_g x))

    @property
    def tokens(self) -> int:
        """T: tokens per frame block = action + state + P patches."""
        return self.patch_tokens + 2

    @property
    def head_dim(self) -> int:
        return self.width // self.heads


@dataclasses.dataclass(frozen=True)
class CemConfig:
    """One CEM planning workload: B problems, N candidates, K elites, R rounds, horizon H."""

    predictor: PredictorConfig
    B: int
    N: int
    K: int
    rounds: int
    horizon: int
    seed: int = 42


TINY = PredictorConfig("tiny", layers=2, width=128, heads=4, mlp=512,
                       patch_tokens=16, embed_dim=64, precision="fp32")
SMALL = PredictorConfig("small", layers=6, width=384, heads=6, mlp=1536,
                        patch_tokens=64, embed_dim=256, precision="bf16")
FULL = PredictorConfig("full", layers=24, width=1024, heads=16, mlp=4096,
                       patch_tokens=256, embed_dim=1408, precision="bf16")

# Gated-MLP variants (the Realtime-VLA notes' FFN: FC1(x) * GELU(FC2(x))) with the same
# hidden width m as their GELU counterparts.
TINY_GATED = dataclasses.replace(TINY, name="tiny_gated", mlp_kind="gated")
SMALL_GATED = dataclasses.replace(SMALL, name="small_gated", mlp_kind="gated")
FULL_GATED = dataclasses.replace(FULL, name="full_gated", mlp_kind="gated")

# Low-precision variants: the same predictors with their LayerNorm-fed GEMMs in fp8 e4m3.
SMALL_FP8 = dataclasses.replace(SMALL, name="small_fp8", precision="fp8")
FULL_FP8 = dataclasses.replace(FULL, name="full_fp8", precision="fp8")
SMALL_GATED_FP8 = dataclasses.replace(SMALL_GATED, name="small_gated_fp8", precision="fp8")

PRESETS: Dict[str, PredictorConfig] = {c.name: c for c in (TINY, SMALL, FULL, TINY_GATED,
                                                            SMALL_GATED, FULL_GATED, SMALL_FP8,
                                                            FULL_FP8, SMALL_GATED_FP8)}

WORKLOADS: Dict[str, CemConfig] = {
    "tiny": CemConfig(TINY, B=1, N=64, K=8, rounds=2, horizon=1),
    "small": CemConfig(SMALL, B=1, N=200, K=20, rounds=5, horizon=2),
    "full": CemConfig(FULL, B=1, N=800, K=80, rounds=10, horizon=1),
    "multistep": CemConfig(FULL, B=1, N=800, K=80, rounds=10, horizon=3),
    "tiny_gated": CemConfig(TINY_GATED, B=1, N=64, K=8, rounds=2, horizon=1),
    "small_gated": CemConfig(SMALL_GATED, B=1, N=200, K=20, rounds=5, horizon=2),
    "full_gated": CemConfig(FULL_GATED, B=1, N=800, K=80, rounds=10, horizon=1),
    "small_fp8": CemConfig(SMALL_FP8, B=1, N=200, K=20, rounds=5, horizon=2),
    "full_fp8": CemConfig(FULL_FP8, B=1, N=800, K=80, rounds=10, horizon=1),
}
for _n in (100, 200, 400, 800, 1600, 3200):
    for _b in (1, 4, 8):
        WORKLOADS[f"sweep_N{_n}_B{_b}"] = CemConfig(FULL, B=_b, N=_n, K=_n // 10,
                                                   rounds=10, horizon=1)


def weight_names(cfg: PredictorConfig) -> List[str]:
    """Canonical tensor order (the weight-blob order of the C ABI)."""
    names = ["W_in", "b_in", "W_a", "b_a", "W_s", "b_s", "pos"]
    for l in range(cfg.layers):
        names += [f"l{l}.{n}" for n in ("ln1_g", "ln1_b", "W_qkv", "b_qkv", "W_o", "b_o",
                                         "ln2_g", "ln2_b", "W_1", "b_1")]
        if cfg.mlp_kind == "gated":
            names += [f"l{l}.W_g", f"l{l}.b_g"]
        names += [f"l{l}.W_2", f"l{l}.b_2"]
    names += ["lnf_g", "lnf_b", "W_out", "b_out"]
    return names


def weight_shapes(cfg: PredictorConfig) -> Dict[str, tuple]:
    """Shapes in the [out, in] convention of a linear layer."""
    d, m, E, A, S, T = cfg.width, cfg.mlp, cfg.embed_dim, cfg.action_dim, cfg.state_dim, cfg.tokens
    shapes = {"W_in": (d, E), "b_in": (d,), "W_a": (d, A), "b_a": (d,), "W_s": (d, S),
              "b_s": (d,), "pos": (T, d)}
    for l in range(cfg.layers):
        shapes.update({f"l{l}.ln1_g": (d,), f"l{l}.ln1_b": (d,), f"l{l}.W_qkv": (3 * d, d),
                       f"l{l}.b_qkv": (3 * d,), f"l{l}.W_o": (d, d), f"l{l}.b_o": (d,),
                       f"l{l}.ln2_g": (d,), f"l{l}.ln2_b": (d,), f"l{l}.W_1": (m, d),
                       f"l{l}.b_1": (m,), f"l{l}.W_2": (d, m), f"l{l}.b_2": (d,)})
        if cfg.mlp_kind == "gated":
            shapes.update({f"l{l}.W_g": (m, d), f"l{l}.b_g": (m,)})
    shapes.update({"lnf_g": (d,), "lnf_b": (d,), "W_out": (E, d), "b_out": (E,)})
    return shapes


LN_GAINS = ("ln1_g", "ln2_g", "lnf_g")


def make_weights(cfg: PredictorConfig, seed: int = 0, std: float = 0.02) -> Dict[str, np.ndarray]:
    """Random-init predictor weights (fp32), drawn in canonical order from one stream."""
    rng = np.random.default_rng(seed)
    shapes = weight_shapes(cfg)
    out: Dict[str, np.ndarray] = {}
    for name in weight_names(cfg):
        w = rng.standard_normal(shapes[name], dtype=np.float32) * np.float32(std)
        if name.split(".")[-1] in LN_GAINS:          # LayerNorm gains near 1
            w = w + np.float32(1.0)
        out[name] = w.astype(np.float32)
    return out


def make_problems(cfg: PredictorConfig, B: int, seed_base: int = 1000):
    """z0, goal [B, P, E] ~ N(0,1) and state0 [B, S] = 0.1 N(0,1); problem b uses seed_base + b."""
    P, E, S = cfg.patch_tokens, cfg.embed_dim, cfg.state_dim
    z0 = np.empty((B, P, E), np.float32)
    goal = np.empty((B, P, E), np.float32)
    s0 = np.empty((B, S), np.float32)
    for b in range(B):
        rng = np.random.default_rng(seed_base + b)
        z0[b] = rng.standard_normal((P, E), dtype=np.float32)
        goal[b] = rng.standard_normal((P, E), dtype=np.float32)
        s0[b] = np.float32(0.1) * rng.standard_normal(S, dtype=np.float32)
    return z0, goal, s0


def make_gaussian(cfg: PredictorConfig, B: int, H: int, mu: float = 0.0, sigma: float = 1.0):
    """Initial CEM Gaussian: mu0, sigma0 [B, H, A]."""
    A = cfg.action_dim
    return (np.full((B, H, A), mu, np.float32), np.full((B, H, A), sigma, np.float32))


def make_actions(cfg: PredictorConfig, B: int, N: int, H: int, seed: int = 7):
    """Action sequences [B, N, H, A] uniform in [-1, 1] (for predictor-only tests)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(-1.0, 1.0, size=(B, N, H, cfg.action_dim)).astype(np.float32)
