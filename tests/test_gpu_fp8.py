"""Low-precision (fp8 e4m3) mode on the GPU against the oracle: the row quantiser bit for
bit (codes are decided in fp32 on both sides), the kind::f8f6f4 GEMM against its definition
on the same codes, and the fp8 predictor's energies against the oracle's fp8 mode."""
import numpy as np
import pytest
import torch

from cem_search_transformer_gb300 import synthetic
from gpu_helpers import (TOL_BF16_ENERGY_REL, cuda, host, make_planner, oracle_weights_for,
                         rel_err)
from oracle import predictor, quant

pytestmark = pytest.mark.gpu

E4M3 = getattr(torch, "float8_e4m3fn", None)
needs_fp8 = pytest.mark.skipif(E4M3 is None, reason="torch without float8_e4m3fn")


@pytest.fixture(scope="module")
def planner():
    p = make_planner("small_fp8", max_horizon=2)
    yield p
    p.close()


def _codes(values):
    """uint8 encodings of e4m3-representable values."""
    return torch.from_numpy(np.asarray(values, np.float32)).to(E4M3).view(torch.uint8)


def _decode(codes_u8):
    return codes_u8.view(E4M3).to(torch.float64).cpu().numpy()


@needs_fp8
def test_quantize_rows_bit_exact(planner):
    rng = np.random.default_rng(0)
    rows, cols = 67, 1000
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x *= np.exp2(rng.uniform(-20, 20, (rows, 1))).astype(np.float32)   # wide row magnitudes
    x[5] = 0.0                                                       # zero row: scale 1
    x[9, :7] = [448.0, -1e-30, 3e-3, 1e6, -2.5, 0.0, 7.0]
    codes = torch.zeros(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(rows, device="cuda")
    planner.quantize_rows_fp8(cuda(x), rows, cols, codes, scales)
    planner.sync_check()
    q_ref, s_ref = quant.quantize_rows(x)
    assert np.array_equal(_decode(codes), q_ref)
    assert np.array_equal(host(scales).astype(np.float64), s_ref)


@needs_fp8
@pytest.mark.parametrize("M,N,K,gelu", [(300, 384, 256, 0),     # 1-CTA, BN = 128, ragged M
                                        (1000, 3072, 1024, 0),  # QKV shape: CTA pairs
                                        (129, 1408, 1024, 0),   # projection to E: 11 tiles
                                        (777, 1536, 384, 1),    # MLP up with GELU
                                        (600, 1024, 384, 2),    # gated pair
                                        (64, 256, 4096, 0)])    # long K
def test_linear_fp8_matches_definition(planner, M, N, K, gelu):
    rng = np.random.default_rng(M + N + K + gelu)
    qa, sa = quant.quantize_rows(rng.standard_normal((M, K)))
    qw, sw = quant.quantize_rows(rng.standard_normal((N, K)) * 0.05)
    bias = rng.standard_normal(N).astype(np.float32) * 0.1
    n_out = N // 2 if gelu == 2 else N
    out = torch.zeros(M, n_out, device="cuda")
    planner.linear_fp8(_codes(qa).cuda(), cuda(sa.astype(np.float32)), _codes(qw).cuda(),
                       cuda(sw.astype(np.float32)), cuda(bias), M, N, K, gelu, out)
    planner.sync_check()
    acc = (qa @ qw.T) * sa[:, None] * sw[None, :] + bias
    if gelu == 1:
        ref = predictor.gelu(acc)
    elif gelu == 2:   # interleaved blocks of 32: FC1 block p, then its gate block
        f = acc.reshape(M, N // 64, 2, 32)
        ref = (f[:, :, 0, :] * predictor.gelu(f[:, :, 1, :])).reshape(M, n_out)
    else:
        ref = acc
    got = host(out)
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(got - ref)) < 2e-5 * scale, np.max(np.abs(got - ref)) / scale


@pytest.mark.parametrize("name,B,N,H", [("small_fp8", 2, 24, 2), ("small_gated_fp8", 1, 16, 2)])
def test_fp8_predictor_matches_oracle(name, B, N, H):
    """Whole predictor in fp8 mode against the oracle's fp8 mode. The LayerNorm outputs are
    quantised from values that differ slightly between the fp32 GPU stream and the fp64
    oracle stream, so single codes can differ by one e4m3 step (6 %), and the random-init
    network amplifies such flips: in the oracle alone, scaling the context frame by 1 + 1e-6
    moves the fp8 frame by ~6 % (GELU MLP) and ~5 % (gated MLP), against ~1e-6 in bf16.
    The frame is therefore held to twice that measured sensitivity (at least 10 %), and the
    energies, averaged over P x E entries, keep the bf16 tolerance."""
    pc = synthetic.PRESETS[name]
    p = make_planner(name, max_horizon=2)
    z0, goal, s0 = synthetic.make_problems(pc, B, seed_base=2011)
    acts = synthetic.make_actions(pc, B, N, H, seed=13)
    zp = torch.zeros(B, N, pc.patch_tokens, pc.embed_dim, device="cuda")
    en = torch.zeros(B, N, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), B, N, H, goal=cuda(goal), z_pred=zp,
                        energy=en)
    p.sync_check()
    zp, en = host(zp), host(en)
    w = oracle_weights_for(name)
    for b in range(B):
        a = acts[b].astype(np.float64)
        z = predictor.rollout(w, pc, z0[b], s0[b], a)[-1]
        e_ref = predictor.energy_l1(z, goal[b])
        assert rel_err(en[b], e_ref) < TOL_BF16_ENERGY_REL
        zpert = predictor.rollout(w, pc, z0[b] * (1 + 1e-6), s0[b], a[:2])[-1]
        sens = np.linalg.norm(zpert - z[:2]) / np.linalg.norm(z[:2])
        zl2 = np.linalg.norm(zp[b] - z) / np.linalg.norm(z)
        print(f"{name} b={b}: energy rel err {rel_err(en[b], e_ref):.2e}, z rel L2 err {zl2:.2e}, "
              f"oracle sensitivity {sens:.2e}")
        assert zl2 < max(0.1, 2 * sens)
    p.close()


def test_full_fp8_sampled_candidates():
    pc = synthetic.FULL_FP8
    p = make_planner("full_fp8", max_horizon=1)
    z0, goal, s0 = synthetic.make_problems(pc, 1)
    acts = synthetic.make_actions(pc, 1, 800, 1, seed=14)
    en = torch.zeros(1, 800, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), 1, 800, 1, goal=cuda(goal), energy=en)
    p.sync_check()
    en = host(en)[0]
    idx = np.array([2, 555])
    z = predictor.rollout(oracle_weights_for("full_fp8"), pc, z0[0], s0[0],
                          acts[0][idx].astype(np.float64))[-1]
    e_ref = predictor.energy_l1(z, goal[0])
    assert rel_err(en[idx], e_ref) < TOL_BF16_ENERGY_REL and np.all(np.isfinite(en))
    print(f"full_fp8: energy rel err {rel_err(en[idx], e_ref):.2e}")
    p.close()


def _energies(name, z0, goal, s0, acts):
    B, N, H, _ = acts.shape
    p = make_planner(name, max_horizon=H)
    en = torch.zeros(B, N, device="cuda")
    p.predictor_forward(cuda(z0), cuda(s0), cuda(acts), B, N, H, goal=cuda(goal), energy=en)
    p.sync_check()
    p.close()
    return host(en)[0].astype(np.float64)


def test_fp8_energy_correlation_reachable_goal():
    """Quality of the fp8 mode as the pages measure their bf16 path: the Pearson correlation
    of candidate energies with the reference (bf16 oracle). With the synthetic recipe's
    independent N(0,1) goal no action gets near the goal and energies differ by ~1e-4
    relative across candidates, below fp8 noise; here the goal is the oracle's own predicted
    frame for a hidden action sequence, so energies spread by ~15 % and rank candidates by
    how close they come. Small configuration, all candidates against the oracle; full shape,
    fp8 against bf16 on the GPU. Measured: bf16 0.9996 and fp8 0.88 (small, 6 layers); fp8
    0.63 against bf16 at full shape (24 layers). The thresholds guard these values."""
    pc = synthetic.SMALL
    z0, _, s0 = synthetic.make_problems(pc, 1)
    w = oracle_weights_for("small")
    astar = synthetic.make_actions(pc, 1, 1, 2, seed=99)[0].astype(np.float64)
    goal = predictor.rollout(w, pc, z0[0], s0[0], astar)[-1][0][None].astype(np.float32)
    acts = synthetic.make_actions(pc, 1, 64, 2, seed=21)
    e_ref = predictor.energy_l1(predictor.rollout(w, pc, z0[0], s0[0], acts[0].astype(np.float64))[-1],
                                goal[0])
    e_bf = _energies("small", z0, goal, s0, acts)
    e_f8 = _energies("small_fp8", z0, goal, s0, acts)
    r_bf, r_f8 = np.corrcoef(e_bf, e_ref)[0, 1], np.corrcoef(e_f8, e_ref)[0, 1]
    print(f"small, reachable goal: spread {e_ref.std() / e_ref.mean():.3f}; Pearson r vs bf16 "
          f"oracle: bf16 {r_bf:.5f}, fp8 {r_f8:.4f}")
    assert r_bf > 0.999 and r_f8 > 0.8

    pf = synthetic.FULL
    z0f, _, s0f = synthetic.make_problems(pf, 1)
    astar = synthetic.make_actions(pf, 1, 1, 1, seed=99)[0].astype(np.float64)
    goalf = predictor.rollout(oracle_weights_for("full"), pf, z0f[0], s0f[0], astar)[-1][0][None]
    goalf = goalf.astype(np.float32)
    actsf = synthetic.make_actions(pf, 1, 800, 1, seed=22)
    e_bf = _energies("full", z0f, goalf, s0f, actsf)
    e_f8 = _energies("full_fp8", z0f, goalf, s0f, actsf)
    r = np.corrcoef(e_bf, e_f8)[0, 1]
    print(f"full, reachable goal: spread {e_bf.std() / e_bf.mean():.3f}; Pearson r fp8 vs bf16 "
          f"(GPU, 800 candidates): {r:.4f}")
    assert r > 0.5          # measured 0.63: e4m3 noise accumulates over 24 layers
