"""8-bit (fp8 e4m3) quantisation of the predictor's large GEMM operands.

Test infrastructure (see the package docstring). The planning page's section "Further
Optimization", part D, names quantising the predictor as the way to shrink the compute term
itself, and the Realtime-VLA notes (section 9.1) point at 8-bit quantisation; neither fixes
a format. Readings taken:

  * format: OCP fp8 E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    no infinities, largest finite 448, smallest subnormal 2^-9), round to nearest even,
    saturating to +-448;
  * weights: one scale per output channel (row of W): s = max |W[n, :]| / 448, codes
    e4m3(W[n, :] / s) (a zero row keeps s = 1);
  * activations: one scale per row (token), s = max |h[r, :]| / 448, computed from the
    LayerNorm output that feeds the GEMM (the only producers that see whole rows);
  * which GEMMs: those fed by a LayerNorm, i.e. QKV, the MLP up-projection (both branches
    when gated) and the projection to the embedding; the attention out-projection and the
    MLP down-projection keep bf16 operands (their inputs are produced tile by tile, so no
    per-row scale exists without another pass), as do the in-projection of z and the
    action / state embeddings;
  * the product of two codes is exact in fp32 and the GEMM accumulates in fp32; the result
    is multiplied by s_row * s_col before the bias;
  * a code is an integer decided by floating point, so it is decided in the CUDA path's
    precision: the row maximum, the factor 448 / max and the scaled value are fp32
    (each operation rounded), then rounded to e4m3; the scale is max / 448 in fp32.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # smallest normal 2^-6
E4M3_MANTISSA_BITS = 3


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturated to +-448; returned as float64."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)   # binade exponent (subnormals share -6)
    quantum = np.ldexp(1.0, e - E4M3_MANTISSA_BITS)
    r = np.round(a / quantum) * quantum       # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(a == 0, 0.0, np.copysign(r, x))


def quantize_rows(a: np.ndarray):
    """Per-row scaled e4m3: returns (codes as float64 values, scales [rows] as float64)."""
    a32 = np.asarray(a, np.float64).astype(np.float32)
    amax = np.max(np.abs(a32), axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1))
    inv = np.where(nz, np.float32(E4M3_MAX) / safe, np.float32(1)).astype(np.float32)
    v = (a32 * inv[..., None]).astype(np.float32)
    s = np.where(nz, safe / np.float32(E4M3_MAX), np.float32(1)).astype(np.float32)
    return round_to_e4m3(v), s.astype(np.float64)


def fake_quant_rows(a: np.ndarray) -> np.ndarray:
    """The values an fp8 operand carries: codes times their row scale."""
    q, s = quantize_rows(a)
    return q * s[..., None]
