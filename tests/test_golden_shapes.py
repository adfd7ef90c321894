"""The synthetic full-shape workload reproduces the data sizes the planning page states."""
import json
import os

from cem_search_transformer_gb300 import synthetic

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_shape_pins.json")))


def test_latent_bytes_match_page():
    cfg = synthetic.FULL
    latents = 2 * cfg.patch_tokens * cfg.embed_dim * 4
    assert abs(latents / GOLD["latents_bytes_stated"] - 1) < GOLD["relative_tolerance"]


def test_action_bytes_per_shard_match_page():
    cfg = synthetic.FULL
    per_shard = GOLD["candidates"] // GOLD["replicas"] * GOLD["horizon"] * cfg.action_dim * 4
    assert abs(per_shard / GOLD["actions_bytes_per_shard_stated"] - 1) < GOLD["relative_tolerance"]


def test_full_predictor_is_about_300M_parameters():
    cfg = synthetic.FULL
    n = sum(int(__import__("numpy").prod(s)) for s in synthetic.weight_shapes(cfg).values())
    assert 2.9e8 < n < 3.2e8
