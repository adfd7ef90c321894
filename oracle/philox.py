"""Candidate sampler: Philox4x32-10 counter-based generator + Box-Muller.

Test infrastructure (see the package docstring). Written from the published
definition of Philox (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
Easy as 1, 2, 3", SC'11): a 4x32-bit counter and a 2x32-bit key, ten rounds of
two 32x32->64 multiplies with the key bumped by the Weyl constants between rounds.

The planning page says only that CEM samples its candidates from a Gaussian
around the current guess (section "Where the sixteen seconds actually
goes") and that a given seed yields the same plan whatever the number of GPUs
(section "Measured on 8x A100"). Reading taken (ours): every draw is addressed by
(candidate n, problem b, round r, quad q) so no draw depends on how candidates
are batched or sharded:

  key     = (seed mod 2^32, seed >> 32)
  counter = (n, b, r*Q + q, 0),  Q = ceil(H*A / 4),  q = (h*A + j) // 4
  u_i     = ((x_i >> 9) + 0.5) * 2^-23           (in (0, 1), exact in f32/f64)
  (z0, z1) = sqrt(-2 ln u0) * (cos 2 pi u1, sin 2 pi u1); same for (u2, u3) -> (z2, z3)
  eps[n, h, j] = z[(h*A + j) mod 4]
  a = clip(mu + sigma * eps, -1, 1)
"""
from __future__ import annotations

import numpy as np

# Philox4x32 multipliers and Weyl key increments (Salmon et al., SC'11).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox rounds on broadcastable uint32 counter words; returns four uint64 arrays < 2^32."""
    x0, x1, x2, x3 = (np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3))
    key0, key1 = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    for _ in range(10):
        p0 = m0 * x0          # < 2^64, exact in uint64
        p1 = m1 * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        x0, x1, x2, x3 = (hi1 ^ x1 ^ np.uint64(key0), lo1,
                          hi0 ^ x3 ^ np.uint64(key1), lo0)
        key0 = (key0 + PHILOX_W0) & 0xFFFFFFFF
        key1 = (key1 + PHILOX_W1) & 0xFFFFFFFF
    return x0, x1, x2, x3


def uniform_open01(x):
    """Map a 32-bit word to (0, 1): top 23 bits plus a half step, scaled by 2^-23."""
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * (2.0 ** -23)


def box_muller(u0, u1):
    """Two independent N(0,1) draws from two uniforms in (0, 1)."""
    r = np.sqrt(-2.0 * np.log(u0))
    theta = 2.0 * np.pi * u1
    return r * np.cos(theta), r * np.sin(theta)


def sample_eps(seed: int, b: int, r: int, N: int, H: int, A: int) -> np.ndarray:
    """Standard normal draws eps[n, h, j] for problem b, round r (float64, [N, H, A])."""
    Q = (H * A + 3) // 4
    k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    n = np.arange(N, dtype=np.uint64)[:, None]
    q = np.arange(Q, dtype=np.uint64)[None, :]
    words = philox4x32_10(n, np.uint64(b), np.uint64(r * Q) + q, np.uint64(0), k0, k1)
    u = [uniform_open01(w) for w in words]              # each [N, Q]
    z0, z1 = box_muller(u[0], u[1])
    z2, z3 = box_muller(u[2], u[3])
    z = np.stack([z0, z1, z2, z3], axis=-1).reshape(N, Q * 4)   # element e -> quad e//4, word e%4
    return z[:, : H * A].reshape(N, H, A)


def sample_actions(mu: np.ndarray, sigma: np.ndarray, eps: np.ndarray) -> np.ndarray:
    """a = clip(mu + sigma * eps, -1, 1); mu, sigma [H, A], eps [N, H, A] (float64)."""
    a = np.asarray(mu, np.float64)[None] + np.asarray(sigma, np.float64)[None] * eps
    return np.clip(a, -1.0, 1.0)
