"""FLOP accounting behind the benchmark's roofline figures, checked against closed forms
written out per matrix product of the predictor (no GPU).

One candidate rollout of the full-shape predictor (L = 24, d = 1024, m = 4096, T = 258,
P = 256, E = 1408) per frame k of the horizon: per layer the QKV product (T x d x 3d), the
attention out-projection (T x d x d), the MLP up and down products (T x d x m each), and
attention over the (k + 1) T cached keys (Q K^T and P V, T x (k+1)T x d each); then the
projection of the P patch rows to E (P x d x E). Every multiply-add counts 2 FLOPs.
"""
import pytest

import bench
from cem_search_transformer_gb300 import synthetic

L, d, m, T, P, E = 24, 1024, 4096, 258, 256, 1408


def test_full_shape_matrix_products_per_rollout():
    pc = synthetic.PRESETS["full"]
    f8, f16 = bench.fp8_flop_split(pc, 1)
    per_layer = 2 * T * d * 3 * d + 2 * T * d * d + 2 * 2 * T * d * m
    assert f8 + f16 == L * per_layer + 2 * P * d * E
    assert abs((f8 + f16) / 1e9 - 156.565) < 0.001
    # the e4m3 share: QKV, MLP up and the projection to E
    assert f8 == L * (2 * T * d * 3 * d + 2 * T * d * m) + 2 * P * d * E


@pytest.mark.parametrize("H", [1, 2, 3])
def test_attention_flops_grow_with_the_cached_frames(H):
    pc = synthetic.PRESETS["full"]
    per_frame = [L * 2 * 2 * T * (k + 1) * T * d for k in range(H)]
    assert bench.attention_flops(pc, H) == sum(per_frame)


def test_full_rollout_total_with_context_projection():
    """GEMMs + attention + the in-projection of the context frame (P x E x d, counted once per
    rollout here) give about 163.8 GFLOP for one full-shape rollout at horizon 1."""
    pc = synthetic.PRESETS["full"]
    f8, f16 = bench.fp8_flop_split(pc, 1)
    total = f8 + f16 + bench.attention_flops(pc, 1) + 2 * P * E * d
    assert abs(total / 1e9 - 163.847) < 0.001


def test_gated_mlp_doubles_the_up_projection():
    f8g, f16g = bench.fp8_flop_split(synthetic.PRESETS["full_gated"], 1)
    f8, f16 = bench.fp8_flop_split(synthetic.PRESETS["full"], 1)
    assert (f8g + f16g) - (f8 + f16) == L * 2 * T * d * m


def test_step_roofline_times_and_fractions():
    pc = synthetic.PRESETS["full"]
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    rollouts = 800 * 10
    f8, f16 = bench.fp8_flop_split(pc, 1)
    flops = (f8 + f16 + bench.attention_flops(pc, 1)) * rollouts
    r = bench.step_roofline(pc, 1, rollouts, None, 1000.0, peaks)
    assert r["tflop_per_step"] == pytest.approx(flops / 1e12)
    assert r["ms_at_measured_burst"] == pytest.approx(flops / 2000e12 * 1e3)
    assert r["ms_at_measured_sustained"] == pytest.approx(flops / 1600e12 * 1e3)
    assert r["ms_at_nominal_dense"] == pytest.approx(flops / 2250e12 * 1e3)
    assert r["frac_of_measured_burst"] == pytest.approx(r["ms_at_measured_burst"] / 1000.0)
    # a measured GEMM count replaces the analytic one; attention is added on top
    gemm_tflop = 1.01 * (f8 + f16) * rollouts / 1e12
    r2 = bench.step_roofline(pc, 1, rollouts, gemm_tflop, 1000.0, peaks)
    assert r2["tflop_per_step"] == pytest.approx(gemm_tflop + bench.attention_flops(pc, 1) * rollouts / 1e12)


def test_fp8_step_roofline_counts_e4m3_products_at_twice_the_rate():
    pc = synthetic.PRESETS["full_fp8"]
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    f8, f16 = bench.fp8_flop_split(pc, 1)
    att = bench.attention_flops(pc, 1)
    r = bench.step_roofline(pc, 1, 1, None, 1.0, peaks)
    assert r["ms_at_measured_burst"] == pytest.approx((f8 / 4000e12 + (f16 + att) / 2000e12) * 1e3)


def test_committed_gemm_traffic_belongs_to_the_committed_kernels():
    """The DRAM traffic bench.py reports for the GEMMs was counted on the kernels whose
    source it names; an edit of that source without new counters (or without a statement
    that the counted kernels are unchanged) makes the bench line report no traffic."""
    assert bench.gemm_source_sha() == bench.GEMM_TRAFFIC_SOURCE_SHA
    assert len(bench.GEMM_DRAM_BYTES_PER_LAUNCH_FULL) == 4
    assert all(1e9 < b < 4e9 for b in bench.GEMM_DRAM_BYTES_PER_LAUNCH_FULL)
