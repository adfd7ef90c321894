"""CPU oracle for one CEM planning step over an action-conditioned JEPA predictor.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA path; both take their inputs from ``cem_search_transformer_gb300.synthetic``
(random draws only) and the oracle computes everything else itself.

The oracle is plain numpy in float64 (library matmul/erf as primitives, no
blocking or fusion), written step by step from "Real-time inference for JEPA
world-model architectures with Ray" (section "Where the sixteen seconds actually
goes"): sample action sequences from a Gaussian, predict where each leads,
measure the distance of each prediction to the goal embedding, refit the Gaussian
to the K closest, and after R rounds hand back the first action of the closest
final-round sequence. Where the page is silent the module docstrings state the
reading taken.

Modules:
  philox     counter-based Philox4x32-10 + Box-Muller candidate sampler
  predictor  pre-LN block-causal transformer predictor, rollout, L1 energy
  cem        elite selection, Gaussian refit, the round loop, warm start, closed loop
  quant      fp8 e4m3 quantisation of the LayerNorm-fed GEMMs (low-precision mode)

Pins (tests/test_oracle_*.py): cuRAND's host Philox4_32_10 stream, hand-derived
Box-Muller closed forms, torch.nn.TransformerEncoderLayer / layer_norm / gelu,
brute-force per-token attention loops, block-causality and permutation
invariants, brute-force sort for top-K, closed-form refit moments, and CEM
convergence to the closed-form optimum of a linear-quadratic problem.
"""
from . import philox, quant, predictor, cem  # noqa: F401
