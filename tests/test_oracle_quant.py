"""Pins for the oracle's fp8 (e4m3) quantiser against torch's float8_e4m3fn conversion,
its fixed points and closed forms of the per-row scaling (CPU only)."""
import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from oracle import predictor, quant

E4M3 = getattr(torch, "float8_e4m3fn", None)
needs_fp8 = pytest.mark.skipif(E4M3 is None, reason="torch without float8_e4m3fn")


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(E4M3).to(torch.float64).numpy()


@needs_fp8
def test_every_code_is_a_fixed_point():
    vals = torch.arange(256, dtype=torch.uint8).view(E4M3).to(torch.float64).numpy()
    vals = vals[np.isfinite(vals)]
    assert len(vals) == 254                              # 0x7F and 0xFF are NaN
    assert np.array_equal(quant.round_to_e4m3(vals), vals)
    assert vals.max() == 448.0 and np.min(vals[vals > 0]) == 2.0 ** -9


@needs_fp8
def test_rounding_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-12, 9, 200000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(quant.round_to_e4m3(x), _torch_e4m3(x))


@needs_fp8
def test_midpoints_round_to_even_like_torch():
    vals = torch.arange(128, dtype=torch.uint8).view(E4M3).to(torch.float64).numpy()
    vals = np.sort(vals[np.isfinite(vals)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)     # exact in fp32
    got = quant.round_to_e4m3(mids)
    assert np.array_equal(got, _torch_e4m3(mids))
    assert np.array_equal(quant.round_to_e4m3(-mids), -got)
    # a tie goes to the value whose mantissa is even: e.g. 1.0625 (between 1 and 1.125) -> 1
    assert quant.round_to_e4m3(np.array([1.0625, 1.1875]))[0] == 1.0
    assert quant.round_to_e4m3(np.array([1.1875]))[0] == 1.25


def test_saturation_and_zero():
    got = quant.round_to_e4m3(np.array([448.0, 460.0, 500.0, 1e9, -1e9, 0.0, -0.0, 2.0 ** -11]))
    assert list(got[:5]) == [448.0, 448.0, 448.0, 448.0, -448.0]
    assert got[5] == 0.0 and got[6] == 0.0 and got[7] == 0.0    # 2^-11 rounds to zero


def test_row_scaling_closed_forms():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((5, 37))
    q, s = quant.quantize_rows(a)
    assert np.allclose(s, np.max(np.abs(a), axis=1) / 448.0, rtol=1e-7, atol=0)
    assert np.array_equal(np.max(np.abs(q), axis=1), np.full(5, 448.0))   # the row max -> 448
    assert np.array_equal(quant.round_to_e4m3(q), q)                     # codes are e4m3
    # power-of-two scaling moves only the scale
    q2, s2 = quant.quantize_rows(a * 8.0)
    assert np.array_equal(q2, q) and np.array_equal(s2, s * 8.0)
    # a zero row keeps scale 1 and zero codes; a constant row with exact scale is exact
    qz, sz = quant.quantize_rows(np.zeros((1, 4)))
    assert np.array_equal(qz, np.zeros((1, 4))) and sz[0] == 1.0
    c = -448.0 * 2.0 ** -10          # scale 2^-10 and factor 1024 are exact in fp32
    assert np.array_equal(quant.fake_quant_rows(np.full((1, 6), c)), np.full((1, 6), c))
    # the relative error of any non-tiny element is at most half an e4m3 step (2^-4)
    fq = quant.fake_quant_rows(a)
    big = np.abs(a) >= np.max(np.abs(a), axis=1, keepdims=True) / 448.0 * 2.0 ** -6
    assert np.all(np.abs(fq - a)[big] <= np.abs(a)[big] * 2.0 ** -4 + 1e-15)


def test_fp8_weights_and_activation_quantisation_points():
    cfg = synthetic.TINY
    w32 = synthetic.make_weights(cfg)
    w8 = predictor.prepare_weights(w32, "fp8")
    wb = predictor.prepare_weights(w32, "bf16")
    for name in ("l0.W_qkv", "l1.W_1", "W_out"):
        q, s = quant.quantize_rows(w32[name].astype(np.float64))
        assert np.array_equal(w8[name], q * s[:, None])
    for name in ("W_in", "l0.W_o", "l1.W_2"):
        assert np.array_equal(w8[name], wb[name])
    assert np.array_equal(w8["l0.b_qkv"], wb["l0.b_qkv"])
    # the fp8 rollout differs from the bf16 one only through quantisation (small)
    z0, goal, s0 = synthetic.make_problems(cfg, 1)
    acts = synthetic.make_actions(cfg, 1, 3, 1)
    z8 = predictor.rollout(w8, cfg, z0[0], s0[0], acts[0].astype(np.float64))[-1]
    zb = predictor.rollout(wb, cfg, z0[0], s0[0], acts[0].astype(np.float64))[-1]
    rel = np.max(np.abs(z8 - zb)) / np.max(np.abs(zb))
    assert 1e-4 < rel < 0.2
