"""The tensor-core GEMM (tcgen05 + TMA) against a plain matmul on bf16-representable inputs."""
import numpy as np
import pytest
import torch

from gpu_helpers import cuda, host, make_planner
from oracle import predictor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def planner():
    p = make_planner("small", max_horizon=2)
    yield p
    p.close()


def _bf16_bits(x):
    return predictor.round_to_bf16(x).view(np.uint32) >> 16


@pytest.mark.parametrize("M,N,K,gelu", [(300, 384, 192, 0),      # ragged M, BN=128 path
                                        (1000, 512, 1024, 1),    # BN=256 path, GELU
                                        (129, 1408, 64, 0),      # one K block, 11 N tiles
                                        (4096, 3072, 1024, 0),   # QKV shape, many tiles
                                        (77, 256, 4096, 1)])     # long K
def test_linear_bf16_matches_matmul(planner, M, N, K, gelu):
    rng = np.random.default_rng(M + N + K)
    A = predictor.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = predictor.round_to_bf16((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    bias = rng.standard_normal(N).astype(np.float32)
    At = cuda(_bf16_bits(A).astype(np.int16))
    Wt = cuda(_bf16_bits(W).astype(np.int16))
    out = torch.zeros(M, N, device="cuda")
    planner.linear_bf16(At, Wt, cuda(bias), M, N, K, gelu, out)
    planner.sync_check()
    ref = A.astype(np.float64) @ W.astype(np.float64).T + bias
    if gelu:
        ref = predictor.gelu(ref)
    got = host(out)
    scale = np.sqrt(K) * 0.05 + 1.0
    assert np.max(np.abs(got - ref)) < 2e-5 * scale * 10, np.max(np.abs(got - ref))


def test_gelu_epilogue_against_exact_erf(planner):
    """GELU of the GEMM epilogue (erf by Abramowitz & Stegun 7.1.26) against the exact-erf
    GELU: with W = I the output is gelu(A) for bf16-representable A over [-8, 8]."""
    K = N = 64
    M = 2048
    x = np.linspace(-8, 8, M * K).astype(np.float32).reshape(M, K)
    A = predictor.round_to_bf16(x)
    W = np.eye(N, K, dtype=np.float32)
    out = torch.zeros(M, N, device="cuda")
    planner.linear_bf16(cuda(_bf16_bits(A).astype(np.int16)), cuda(_bf16_bits(W).astype(np.int16)),
                        None, M, N, K, 1, out)
    planner.sync_check()
    ref = predictor.gelu(A.astype(np.float64))
    err = np.abs(host(out) - ref)
    assert np.max(err / np.maximum(1.0, np.abs(ref))) < 2e-6, np.max(err)
