"""Action-conditioned JEPA predictor (V-JEPA2-AC style), rollout and L1 energy.

Test infrastructure (see the package docstring). float64 numpy throughout.

The planning page fixes what the predictor is used for: it is frame-causal
(section "Measured on 8x A100": cached keys and values stay exact between rollout
steps, since the frames already processed do not change), it advances one frame at
a time across the
horizon (section "E. Serving-level optimization"), and each rollout is scored
against the goal embedding (section "Where the sixteen seconds actually goes").
It gives no internals; the shapes come from the synthetic configurations and the
rest is the plainest reading, stated here:

  * tokens of frame block k (T = P + 2 of them): [action a_k, state s_k, P patches of z_k];
    a_k, s_k and z_k are linearly embedded to width d, then pos[t] is added
    (the same positions in every block; no temporal embedding, no RoPE);
  * s_0 = state0 and s_k = s_{k-1} + a_{k-1} (delta actions integrate the state);
  * z_0 = the encoded context frame, z_k = the prediction for k >= 1 (autoregressive);
  * L pre-LN layers: x += W_o Attn(LN1 x) + b_o ; x += W_2 GELU(W_1 LN2 x + b_1) + b_2,
    GELU with erf, LayerNorm eps 1e-5, attention scale 1/sqrt(d/h);
  * gated-MLP variant (the Realtime-VLA notes, section 4.2 "Fusing Gated Linear Layers":
    the up-projection is FC1(x, w1) * GELU(FC2(x, w2))): with FC1 = W_1, b_1 and
    FC2 = W_g, b_g, x += W_2 [(W_1 h + b_1) * GELU(W_g h + b_g)] + b_2, h = LN2 x;
  * block-causal mask: a query in block i sees every key of blocks j <= i;
  * prediction z_{k+1}[p] = W_out LN_f(x at patch p of block k) + b_out;
  * energy = mean over the P x E entries of |z_H - goal| (L1; the mean ranks like the sum).

Each rollout step is a full recompute over blocks 0..k with the mask. That is the
definition; a KV cache reaches the same values because of block causality.

In bf16 mode the matrices that the CUDA path stores in bf16 (W_in, W_qkv, W_o, W_1,
W_g, W_2, W_out) are rounded to bf16 (round to nearest even) before upcasting; all
activations stay float64.

In fp8 mode (``quant.py``) the GEMMs fed by a LayerNorm (QKV, MLP up, projection to E) take
per-channel scaled e4m3 weights and per-row scaled e4m3 copies of the LayerNorm output; the
other matrices are bf16 as in bf16 mode.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np
from scipy.special import erf

from . import quant

MATRIX_SUFFIXES = ("W_in", "W_qkv", "W_o", "W_1", "W_g", "W_2", "W_out")
FP8_SUFFIXES = ("W_qkv", "W_1", "W_g", "W_out")      # fp8 mode: e4m3 with row scales


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned as float32."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32)


def prepare_weights(w: Dict[str, np.ndarray], precision: str) -> Dict[str, np.ndarray]:
    """float64 copies of the fp32 weights; bf16 mode rounds the GEMM matrices first; fp8
    mode quantises the LayerNorm-fed GEMM matrices per output channel instead."""
    out = {}
    for name, v in w.items():
        v = np.asarray(v, np.float32)
        kind = name.split(".")[-1]
        if precision == "fp8" and kind in FP8_SUFFIXES:
            out[name] = quant.fake_quant_rows(v.astype(np.float64))
            continue
        if precision in ("bf16", "fp8") and kind in MATRIX_SUFFIXES:
            v = round_to_bf16(v)
        out[name] = v.astype(np.float64)
    if precision == "fp8":
        out["__fp8__"] = np.ones(1)               # marks the activation quantisation
    return out


def _gemm_input(w: Dict[str, np.ndarray], h: np.ndarray) -> np.ndarray:
    """What a LayerNorm-fed GEMM multiplies: h itself, or in fp8 mode its per-row e4m3 copy."""
    return quant.fake_quant_rows(h) if "__fp8__" in w else h


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis with the biased variance, then gain and shift."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


def gelu(x: np.ndarray) -> np.ndarray:
    """GELU with the exact Gaussian CDF: x * Phi(x)."""
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def block_causal_allowed(n_blocks: int, T: int) -> np.ndarray:
    """allowed[i, j] is True when query token i may attend to key token j (block(j) <= block(i))."""
    blk = np.arange(n_blocks * T) // T
    return blk[None, :] <= blk[:, None]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(hd)) v over allowed keys; q, k, v [..., heads, L, hd]."""
    hd = q.shape[-1]
    s = np.einsum("...qd,...kd->...qk", q, k) / np.sqrt(hd)
    s = np.where(allowed, s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("...qk,...kd->...qd", p, v)


def transformer_layer(x: np.ndarray, w: Dict[str, np.ndarray], l: int, heads: int,
                      allowed: np.ndarray, eps: float) -> np.ndarray:
    """One pre-LN layer on x [n, L, d]."""
    n, L, d = x.shape
    hd = d // heads
    h = _gemm_input(w, layer_norm(x, w[f"l{l}.ln1_g"], w[f"l{l}.ln1_b"], eps))
    qkv = h @ w[f"l{l}.W_qkv"].T + w[f"l{l}.b_qkv"]                  # [n, L, 3d]
    q, k, v = (qkv[..., i * d:(i + 1) * d].reshape(n, L, heads, hd).transpose(0, 2, 1, 3)
               for i in range(3))
    o = attention(q, k, v, allowed).transpose(0, 2, 1, 3).reshape(n, L, d)
    x = x + o @ w[f"l{l}.W_o"].T + w[f"l{l}.b_o"]
    h2 = _gemm_input(w, layer_norm(x, w[f"l{l}.ln2_g"], w[f"l{l}.ln2_b"], eps))
    fc1 = h2 @ w[f"l{l}.W_1"].T + w[f"l{l}.b_1"]
    if f"l{l}.W_g" in w:                                  # gated MLP
        u = fc1 * gelu(h2 @ w[f"l{l}.W_g"].T + w[f"l{l}.b_g"])
    else:
        u = gelu(fc1)
    return x + u @ w[f"l{l}.W_2"].T + w[f"l{l}.b_2"]


def embed_block(w: Dict[str, np.ndarray], z: np.ndarray, a: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Tokens of one frame block: z [n, P, E], a [n, A], s [n, S] -> [n, P + 2, d]."""
    act = a @ w["W_a"].T + w["b_a"]
    st = s @ w["W_s"].T + w["b_s"]
    patches = z @ w["W_in"].T + w["b_in"]
    x = np.concatenate([act[:, None, :], st[:, None, :], patches], axis=1)
    return x + w["pos"][None]


def rollout(w: Dict[str, np.ndarray], cfg, z0: np.ndarray, state0: np.ndarray,
            actions: np.ndarray) -> List[np.ndarray]:
    """Autoregressive rollout of n candidates over the horizon.

    w: prepare_weights output; z0 [P, E]; state0 [S]; actions [n, H, A].
    Returns [z_1, ..., z_H], each [n, P, E] float64.
    """
    n, H, _ = actions.shape
    P, T = cfg.patch_tokens, cfg.tokens
    a = np.asarray(actions, np.float64)
    states = [np.broadcast_to(np.asarray(state0, np.float64), (n, cfg.state_dim))]
    for k in range(1, H):
        states.append(states[-1] + a[:, k - 1])
    frames = [np.broadcast_to(np.asarray(z0, np.float64), (n, P, cfg.embed_dim))]
    preds = []
    for k in range(H):
        x = np.concatenate([embed_block(w, frames[j], a[:, j], states[j]) for j in range(k + 1)],
                           axis=1)                                   # [n, (k+1) T, d]
        allowed = block_causal_allowed(k + 1, T)
        for l in range(cfg.layers):
            x = transformer_layer(x, w, l, cfg.heads, allowed, cfg.ln_eps)
        xp = x[:, k * T + 2:(k + 1) * T]                              # patches of block k
        z_next = _gemm_input(w, layer_norm(xp, w["lnf_g"], w["lnf_b"], cfg.ln_eps)) @ w["W_out"].T \
            + w["b_out"]
        preds.append(z_next)
        frames.append(z_next)
    return preds


def energy_l1(z_pred: np.ndarray, goal: np.ndarray) -> np.ndarray:
    """Mean absolute difference to the goal embedding: z_pred [n, P, E], goal [P, E] -> [n]."""
    diff = np.abs(np.asarray(z_pred, np.float64) - np.asarray(goal, np.float64)[None])
    return diff.reshape(diff.shape[0], -1).mean(axis=1)
