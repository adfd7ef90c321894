"""Pins for the oracle's predictor: library layers, brute-force loops, invariants (CPU only)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from oracle import predictor

MICRO = synthetic.PredictorConfig("micro", layers=2, width=32, heads=4, mlp=64,
                                  patch_tokens=5, embed_dim=12, precision="fp32")


def _w(cfg, seed=0):
    return predictor.prepare_weights(synthetic.make_weights(cfg, seed=seed, std=0.2), "fp32")


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.0e38, -1e-40],
                                 np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(predictor.round_to_bf16(x), ref)


def test_layer_norm_matches_torch():
    rng = np.random.default_rng(1)
    x, g, b = rng.standard_normal((7, 33)), rng.standard_normal(33), rng.standard_normal(33)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (33,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(predictor.layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)
    y = predictor.layer_norm(x, np.ones(33), np.zeros(33), 0.0)
    assert np.allclose(y.mean(-1), 0, atol=1e-12) and np.allclose(y.var(-1), 1, atol=1e-12)


def test_gelu_matches_torch():
    x = np.linspace(-8, 8, 2001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x)).numpy()
    assert np.allclose(predictor.gelu(x), ref, rtol=1e-14, atol=1e-15)


def test_block_causal_mask_brute_force():
    T, nb = 3, 4
    allowed = predictor.block_causal_allowed(nb, T)
    for i in range(nb * T):
        for j in range(nb * T):
            assert allowed[i, j] == ((j // T) <= (i // T))


def test_attention_brute_force_loops():
    rng = np.random.default_rng(2)
    heads, L, hd = 2, 7, 3
    q, k, v = (rng.standard_normal((heads, L, hd)) for _ in range(3))
    allowed = predictor.block_causal_allowed(3, 3)[:L, :L]
    got = predictor.attention(q, k, v, allowed)
    for h in range(heads):
        for i in range(L):
            scores = [sum(q[h, i, t] * k[h, j, t] for t in range(hd)) / math.sqrt(hd)
                      if allowed[i, j] else None for j in range(L)]
            m = max(s for s in scores if s is not None)
            wts = [math.exp(s - m) if s is not None else 0.0 for s in scores]
            z = sum(wts)
            for t in range(hd):
                want = sum(wts[j] * v[h, j, t] for j in range(L)) / z
                assert abs(got[h, i, t] - want) < 1e-12


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((2, 9, 4)) * 5, rng.standard_normal((2, 9, 4)) * 5
    ones = np.ones((2, 9, 1))
    allowed = predictor.block_causal_allowed(3, 3)
    assert np.allclose(predictor.attention(q, k, ones, allowed), 1.0, atol=1e-13)


def test_layer_matches_torch_encoder_layer():
    """A pre-LN layer with the block-causal mask equals torch.nn.TransformerEncoderLayer."""
    cfg = MICRO
    w = _w(cfg, seed=4)
    d, T, nb = cfg.width, cfg.tokens, 3
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, nb * T, d))
    allowed = predictor.block_causal_allowed(nb, T)
    got = predictor.transformer_layer(x, w, 1, cfg.heads, allowed, cfg.ln_eps)
    layer = torch.nn.TransformerEncoderLayer(d, cfg.heads, cfg.mlp, dropout=0.0, activation="gelu",
                                             layer_norm_eps=cfg.ln_eps, batch_first=True,
                                             norm_first=True, dtype=torch.float64)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(t(w["l1.W_qkv"]))
        layer.self_attn.in_proj_bias.copy_(t(w["l1.b_qkv"]))
        layer.self_attn.out_proj.weight.copy_(t(w["l1.W_o"]))
        layer.self_attn.out_proj.bias.copy_(t(w["l1.b_o"]))
        layer.linear1.weight.copy_(t(w["l1.W_1"]))
        layer.linear1.bias.copy_(t(w["l1.b_1"]))
        layer.linear2.weight.copy_(t(w["l1.W_2"]))
        layer.linear2.bias.copy_(t(w["l1.b_2"]))
        layer.norm1.weight.copy_(t(w["l1.ln1_g"]))
        layer.norm1.bias.copy_(t(w["l1.ln1_b"]))
        layer.norm2.weight.copy_(t(w["l1.ln2_g"]))
        layer.norm2.bias.copy_(t(w["l1.ln2_b"]))
        ref = layer(t(x), src_mask=t(~allowed)).numpy()
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-11)


def _torch_layer(w, l, cfg, W1, b1, activation):
    """torch.nn.TransformerEncoderLayer (pre-LN) carrying layer l's weights, with the given
    first MLP linear and activation."""
    layer = torch.nn.TransformerEncoderLayer(cfg.width, cfg.heads, cfg.mlp, dropout=0.0,
                                             activation=activation, layer_norm_eps=cfg.ln_eps,
                                             batch_first=True, norm_first=True,
                                             dtype=torch.float64)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(t(w[f"l{l}.W_qkv"]))
        layer.self_attn.in_proj_bias.copy_(t(w[f"l{l}.b_qkv"]))
        layer.self_attn.out_proj.weight.copy_(t(w[f"l{l}.W_o"]))
        layer.self_attn.out_proj.bias.copy_(t(w[f"l{l}.b_o"]))
        layer.linear1.weight.copy_(t(W1))
        layer.linear1.bias.copy_(t(b1))
        layer.linear2.weight.copy_(t(w[f"l{l}.W_2"]))
        layer.linear2.bias.copy_(t(w[f"l{l}.b_2"]))
        layer.norm1.weight.copy_(t(w[f"l{l}.ln1_g"]))
        layer.norm1.bias.copy_(t(w[f"l{l}.ln1_b"]))
        layer.norm2.weight.copy_(t(w[f"l{l}.ln2_g"]))
        layer.norm2.bias.copy_(t(w[f"l{l}.ln2_b"]))
    return layer


def test_gated_layer_reduces_to_torch_layers():
    """Gated MLP u = (W_1 h + b_1) * GELU(W_g h + b_g), pinned by its two degenerate cases:
    a constant-one linear branch (W_1 = 0, b_1 = 1) leaves a GELU MLP whose first linear is
    the gate (torch's gelu layer), and a constant gate (W_g = 0, b_g = c) leaves a linear MLP
    scaled by GELU(c) (torch's layer with that activation). Applying GELU to the wrong branch,
    dropping a bias or adding instead of multiplying fails one of them."""
    cfg = dataclasses.replace(MICRO, mlp_kind="gated")
    w = _w(cfg, seed=8)
    d, T, nb, l = cfg.width, cfg.tokens, 2, 1
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, nb * T, d))
    allowed = predictor.block_causal_allowed(nb, T)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))

    w1 = dict(w)
    w1[f"l{l}.W_1"] = np.zeros_like(w[f"l{l}.W_1"])
    w1[f"l{l}.b_1"] = np.ones_like(w[f"l{l}.b_1"])
    got = predictor.transformer_layer(x, w1, l, cfg.heads, allowed, cfg.ln_eps)
    layer = _torch_layer(w, l, cfg, w[f"l{l}.W_g"], w[f"l{l}.b_g"], "gelu")
    with torch.no_grad():
        ref = layer(t(x), src_mask=t(~allowed)).numpy()
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-11)

    c = 1.3
    w2 = dict(w)
    w2[f"l{l}.W_g"] = np.zeros_like(w[f"l{l}.W_g"])
    w2[f"l{l}.b_g"] = np.full_like(w[f"l{l}.b_g"], c)
    got = predictor.transformer_layer(x, w2, l, cfg.heads, allowed, cfg.ln_eps)
    g_c = torch.nn.functional.gelu(torch.tensor(c, dtype=torch.float64))
    layer = _torch_layer(w, l, cfg, w[f"l{l}.W_1"], w[f"l{l}.b_1"], lambda u: u * g_c)
    with torch.no_grad():
        ref = layer(t(x), src_mask=t(~allowed)).numpy()
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-11)

    # and the general case differs from both (the gate really multiplies)
    full = predictor.transformer_layer(x, w, l, cfg.heads, allowed, cfg.ln_eps)
    assert not np.allclose(full, got, rtol=1e-6)


def test_gated_weights_in_canonical_order():
    cfg = dataclasses.replace(MICRO, mlp_kind="gated")
    names = synthetic.weight_names(cfg)
    i = names.index("l0.b_1")
    assert names[i + 1:i + 5] == ["l0.W_g", "l0.b_g", "l0.W_2", "l0.b_2"]
    assert synthetic.weight_shapes(cfg)["l0.W_g"] == (cfg.mlp, cfg.width)
    wb = predictor.prepare_weights(synthetic.make_weights(cfg), "bf16")
    assert np.array_equal(wb["l0.W_g"], predictor.round_to_bf16(synthetic.make_weights(cfg)["l0.W_g"]))


@pytest.mark.parametrize("kind", ["gelu", "gated"])
def test_synthetic_weight_recipe(kind):
    """The input recipe: every matrix and bias N(0, 0.02); only the LayerNorm gains are
    1 + N(0, 0.02) (the gate matrix W_g and bias b_g are ordinary weights, not gains)."""
    cfg = dataclasses.replace(synthetic.SMALL, mlp_kind=kind)
    w = synthetic.make_weights(cfg)
    for name, v in w.items():
        v = v.astype(np.float64)
        gain = name.split(".")[-1] in ("ln1_g", "ln2_g", "lnf_g")
        assert abs(v.mean() - (1.0 if gain else 0.0)) < 0.01, name
        assert abs(v.std() - 0.02) < 0.005, name


def _incremental_rollout(w, cfg, z0, s0, actions):
    """Independent KV-cached rollout: each layer attends over cached keys/values of earlier blocks."""
    n, H, _ = actions.shape
    d, hd, T = cfg.width, cfg.head_dim, cfg.tokens
    cache = [[] for _ in range(cfg.layers)]
    z, s, preds = np.broadcast_to(z0, (n,) + z0.shape), np.broadcast_to(s0, (n, len(s0))), []
    for k in range(H):
        x = predictor.embed_block(w, z, actions[:, k], s)
        for l in range(cfg.layers):
            h = predictor.layer_norm(x, w[f"l{l}.ln1_g"], w[f"l{l}.ln1_b"], cfg.ln_eps)
            qkv = h @ w[f"l{l}.W_qkv"].T + w[f"l{l}.b_qkv"]
            cache[l].append(qkv[..., d:])
            kv = np.concatenate(cache[l], axis=1)
            o = np.zeros((n, T, d))
            for hh in range(cfg.heads):
                qh = qkv[..., hh * hd:(hh + 1) * hd]
                kh = kv[..., hh * hd:(hh + 1) * hd]
                vh = kv[..., d + hh * hd:d + (hh + 1) * hd]
                sc = qh @ kh.transpose(0, 2, 1) / math.sqrt(hd)
                p = np.exp(sc - sc.max(-1, keepdims=True))
                o[..., hh * hd:(hh + 1) * hd] = (p / p.sum(-1, keepdims=True)) @ vh
            x = x + o @ w[f"l{l}.W_o"].T + w[f"l{l}.b_o"]
            h2 = predictor.layer_norm(x, w[f"l{l}.ln2_g"], w[f"l{l}.ln2_b"], cfg.ln_eps)
            x = x + predictor.gelu(h2 @ w[f"l{l}.W_1"].T + w[f"l{l}.b_1"]) @ w[f"l{l}.W_2"].T \
                + w[f"l{l}.b_2"]
        z = predictor.layer_norm(x[:, 2:], w["lnf_g"], w["lnf_b"], cfg.ln_eps) @ w["W_out"].T \
            + w["b_out"]
        preds.append(z)
        s = s + actions[:, k]
    return preds


def test_rollout_equals_kv_cached_recurrence():
    cfg = MICRO
    w = _w(cfg, 6)
    rng = np.random.default_rng(7)
    z0, s0 = rng.standard_normal((cfg.patch_tokens, cfg.embed_dim)), rng.standard_normal(7)
    acts = rng.uniform(-1, 1, (3, 3, 7))
    full = predictor.rollout(w, cfg, z0, s0, acts)
    inc = _incremental_rollout(w, cfg, z0, s0, acts)
    for a, b in zip(full, inc):
        assert np.allclose(a, b, rtol=1e-11, atol=1e-12)


def test_rollout_is_causal_in_actions():
    """z_{k+1} depends on a_0..a_k only: changing the last action leaves earlier frames intact."""
    cfg = MICRO
    w = _w(cfg, 8)
    rng = np.random.default_rng(9)
    z0, s0 = rng.standard_normal((cfg.patch_tokens, cfg.embed_dim)), rng.standard_normal(7)
    acts = rng.uniform(-1, 1, (2, 3, 7))
    acts2 = acts.copy()
    acts2[:, 2] += 0.3
    p1, p2 = predictor.rollout(w, cfg, z0, s0, acts), predictor.rollout(w, cfg, z0, s0, acts2)
    assert np.array_equal(p1[0], p2[0]) and np.array_equal(p1[1], p2[1])
    assert not np.allclose(p1[2], p2[2])
    # the state token carries a_0 into block 1: changing a_0 alters z_2 even with W_a = 0
    w0 = dict(w, W_a=np.zeros_like(w["W_a"]))
    acts3 = acts.copy()
    acts3[:, 0] += 0.3
    q1, q3 = predictor.rollout(w0, cfg, z0, s0, acts), predictor.rollout(w0, cfg, z0, s0, acts3)
    assert np.array_equal(q1[0], q3[0]) and not np.allclose(q1[1], q3[1])


def test_candidate_permutation_equivariance():
    cfg = MICRO
    w = _w(cfg, 10)
    rng = np.random.default_rng(11)
    z0, s0 = rng.standard_normal((cfg.patch_tokens, cfg.embed_dim)), rng.standard_normal(7)
    acts = rng.uniform(-1, 1, (6, 2, 7))
    perm = rng.permutation(6)
    a = predictor.rollout(w, cfg, z0, s0, acts)[-1]
    b = predictor.rollout(w, cfg, z0, s0, acts[perm])[-1]
    assert np.allclose(a[perm], b, rtol=1e-13, atol=1e-14)


def test_patch_permutation_equivariance_without_positions():
    """With pos = 0 nothing but token content distinguishes patches: permuting the context
    patches permutes the predicted patches (catches patch/token slicing mistakes)."""
    cfg = MICRO
    w = _w(cfg, 12)
    w["pos"] = np.zeros_like(w["pos"])
    rng = np.random.default_rng(13)
    z0, s0 = rng.standard_normal((cfg.patch_tokens, cfg.embed_dim)), rng.standard_normal(7)
    acts = rng.uniform(-1, 1, (2, 2, 7))
    perm = rng.permutation(cfg.patch_tokens)
    a = predictor.rollout(w, cfg, z0, s0, acts)
    b = predictor.rollout(w, cfg, z0[perm], s0, acts)
    for x, y in zip(a, b):
        assert np.allclose(x[:, perm], y, rtol=1e-11, atol=1e-12)


def test_actions_enter_only_through_action_and_state_tokens():
    cfg = MICRO
    w = _w(cfg, 14)
    w["W_a"] = np.zeros_like(w["W_a"])
    rng = np.random.default_rng(15)
    z0, s0 = rng.standard_normal((cfg.patch_tokens, cfg.embed_dim)), rng.standard_normal(7)
    acts = rng.uniform(-1, 1, (4, 1, 7))
    z = predictor.rollout(w, cfg, z0, s0, acts)[0]
    assert np.allclose(z, z[:1], rtol=0, atol=1e-14)


def test_energy_closed_form():
    rng = np.random.default_rng(16)
    g = rng.standard_normal((5, 6))
    z = np.stack([g + 0.25, g - 0.5, g])
    assert np.allclose(predictor.energy_l1(z, g), [0.25, 0.5, 0.0], atol=1e-15)


def _embed_by_loops(w, z, a, s):
    """Frame-block tokens written out one token and one output channel at a time.

    Token 0 embeds the action, token 1 the state, tokens 2.. embed the P context patches;
    every token then gets the learned position of its index within the block."""
    n, P, E = z.shape
    d = w["pos"].shape[1]
    out = np.zeros((n, P + 2, d))
    for i in range(n):
        for t in range(P + 2):
            for c in range(d):
                if t == 0:
                    v = w["b_a"][c] + sum(w["W_a"][c, j] * a[i, j] for j in range(a.shape[1]))
                elif t == 1:
                    v = w["b_s"][c] + sum(w["W_s"][c, j] * s[i, j] for j in range(s.shape[1]))
                else:
                    v = w["b_in"][c] + sum(w["W_in"][c, e] * z[i, t - 2, e] for e in range(E))
                out[i, t, c] = v + w["pos"][t, c]
    return out


def test_embed_block_equals_per_token_loops():
    """The frame-block embedding against an explicit loop over candidates, tokens and channels
    (a dropped bias, a position added to only some tokens, or swapped action / state slots all
    change some entry)."""
    cfg = synthetic.PredictorConfig("embed", layers=1, width=6, heads=2, mlp=8, patch_tokens=3,
                                    embed_dim=4, precision="fp32")
    w = _w(cfg, seed=20)
    rng = np.random.default_rng(21)
    z = rng.standard_normal((2, cfg.patch_tokens, cfg.embed_dim))
    a, s = rng.uniform(-1, 1, (2, 7)), rng.standard_normal((2, 7))
    got = predictor.embed_block(w, z, a, s)
    assert got.shape == (2, cfg.tokens, cfg.width)
    assert np.allclose(got, _embed_by_loops(w, z, a, s), rtol=1e-13, atol=1e-14)


def test_embed_block_zero_weight_probes():
    """Probes with zeroed parts of the embedding, each isolating one term:
    W_in = W_a = W_s = 0 leaves bias + position per slot; pos = 0 with only one slot's bias
    non-zero lights up exactly that slot; unit inputs read one column of each matrix into
    its own slot, in the order [action, state, patches]."""
    cfg = synthetic.PredictorConfig("embed", layers=1, width=5, heads=1, mlp=4, patch_tokens=2,
                                    embed_dim=3, precision="fp32")
    w = _w(cfg, seed=22)
    rng = np.random.default_rng(23)
    z = rng.standard_normal((1, 2, 3))
    a, s = rng.uniform(-1, 1, (1, 7)), rng.standard_normal((1, 7))
    zero = {k: np.zeros_like(w[k]) for k in ("W_in", "W_a", "W_s")}
    x = predictor.embed_block(dict(w, **zero), z, a, s)[0]
    assert np.allclose(x[0], w["b_a"] + w["pos"][0], atol=1e-15)
    assert np.allclose(x[1], w["b_s"] + w["pos"][1], atol=1e-15)
    for p in range(2):
        assert np.allclose(x[2 + p], w["b_in"] + w["pos"][2 + p], atol=1e-15)
    # one bias at a time, positions and matrices off: only that slot is non-zero
    off = dict(w, **zero, pos=np.zeros_like(w["pos"]),
               b_a=np.zeros_like(w["b_a"]), b_s=np.zeros_like(w["b_s"]), b_in=np.zeros_like(w["b_in"]))
    for name, slots in (("b_a", [0]), ("b_s", [1]), ("b_in", [2, 3])):
        x = predictor.embed_block(dict(off, **{name: np.arange(1.0, 6.0)}), z, a, s)[0]
        for t in range(4):
            assert np.array_equal(x[t], np.arange(1.0, 6.0) if t in slots else np.zeros(5)), (name, t)
    # unit inputs: action e_2 gives column 2 of W_a in slot 0, state e_4 column 4 of W_s in
    # slot 1, and patch p = e_p gives column p of W_in in slot 2 + p
    bare = dict(w, pos=np.zeros_like(w["pos"]), b_a=np.zeros_like(w["b_a"]),
                b_s=np.zeros_like(w["b_s"]), b_in=np.zeros_like(w["b_in"]))
    ea, es, ez = np.zeros((1, 7)), np.zeros((1, 7)), np.zeros((1, 2, 3))
    ea[0, 2], es[0, 4], ez[0, 0, 0], ez[0, 1, 1] = 1.0, 1.0, 1.0, 1.0
    x = predictor.embed_block(bare, ez, ea, es)[0]
    assert np.array_equal(x[0], w["W_a"][:, 2])
    assert np.array_equal(x[1], w["W_s"][:, 4])
    assert np.array_equal(x[2], w["W_in"][:, 0])
    assert np.array_equal(x[3], w["W_in"][:, 1])
