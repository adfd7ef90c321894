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
                                        (4100, 1536, 384, 1),    # GELU on CTA pairs, ragged M,
                                                                 # both accumulators
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
    """GELU of the GEMM epilogue (erf by Abramowitz & Stegun 7.1.28) against the exact-erf
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


def _interleave32(a, b):
    """Rows (or entries) of a and b in alternating blocks of 32: a[0:32], b[0:32], a[32:64], ..."""
    n = a.shape[0]
    out = np.empty((2 * n,) + a.shape[1:], a.dtype)
    for p in range(n // 32):
        out[64 * p:64 * p + 32] = a[32 * p:32 * p + 32]
        out[64 * p + 32:64 * p + 64] = b[32 * p:32 * p + 32]
    return out


@pytest.mark.parametrize("M,n,K", [(300, 128, 192),      # ragged M, one tile of 4 pairs
                                   (1000, 1536, 384),    # small predictor's up-projection
                                   (129, 512, 1024),
                                   (4100, 1536, 384)])   # > 1 tile per CTA, both accumulators
def test_gated_linear_matches_definition(planner, M, n, K):
    """Gated up-projection (FC1 * GELU(gate)) in one GEMM over interleaved weights, against
    the definition computed with the two matrices separately."""
    rng = np.random.default_rng(M + n + K)
    A = predictor.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W1 = predictor.round_to_bf16((rng.standard_normal((n, K)) * 0.05).astype(np.float32))
    Wg = predictor.round_to_bf16((rng.standard_normal((n, K)) * 0.05).astype(np.float32))
    b1 = rng.standard_normal(n).astype(np.float32)
    bg = rng.standard_normal(n).astype(np.float32)
    W = _interleave32(W1, Wg)
    bias = _interleave32(b1, bg)
    out = torch.zeros(M, n, device="cuda")
    planner.linear_bf16(cuda(_bf16_bits(A).astype(np.int16)), cuda(_bf16_bits(W).astype(np.int16)),
                        cuda(bias), M, 2 * n, K, 2, out)
    planner.sync_check()
    A64 = A.astype(np.float64)
    ref = (A64 @ W1.astype(np.float64).T + b1) * predictor.gelu(A64 @ Wg.astype(np.float64).T + bg)
    got = host(out)
    scale = (np.sqrt(K) * 0.05 + 1.0) ** 2
    assert np.max(np.abs(got - ref)) < 2e-5 * scale * 10, np.max(np.abs(got - ref))
    # the wrong pairing (GELU on FC1) is far off: the test can tell the branches apart
    swapped = predictor.gelu(A64 @ W1.astype(np.float64).T + b1) * (A64 @ Wg.astype(np.float64).T + bg)
    assert np.max(np.abs(got - swapped)) > 1e-2


def test_gated_linear_rejects_bad_shapes(planner):
    from cem_search_transformer_gb300.binding import JepaError
    A = torch.zeros(64, 64, dtype=torch.int16, device="cuda")
    W = torch.zeros(384, 64, dtype=torch.int16, device="cuda")
    out = torch.zeros(64, 192, device="cuda")
    bias = torch.zeros(384, device="cuda")
    with pytest.raises(JepaError):
        planner.linear_bf16(A, W, bias, 64, 384, 64, 2, out)      # N not a multiple of 256
    with pytest.raises(JepaError):
        planner.linear_bf16(A, W[:256], None, 64, 256, 64, 2, out)  # gated needs a bias


def _bf16_to_f64(bits):
    """bf16 bit patterns (int16 / uint16 array) as float64 values."""
    return (bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(8000, 1024, 1024),   # CTA pairs: several tiles per pair,
                                                          # both accumulators, ragged last tile
                                   (4100, 768, 256),     # CTA pairs, M not a multiple of 32
                                   (300, 384, 192)])     # single CTAs
def test_linear_resid_matches_matmul(planner, M, N, K):
    """Residual GEMM (attention out-projection / MLP down-projection): x += A W^T + b in fp32,
    against the same sum in float64 on bf16-representable A and W."""
    rng = np.random.default_rng(M + N + K + 1)
    A = predictor.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = predictor.round_to_bf16((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    bias = rng.standard_normal(N).astype(np.float32)
    x0 = rng.standard_normal((M, N)).astype(np.float32)
    x = cuda(x0)
    planner.linear_resid_bf16(cuda(_bf16_bits(A).astype(np.int16)), cuda(_bf16_bits(W).astype(np.int16)),
                              cuda(bias), M, N, K, x)
    planner.sync_check()
    ref = x0.astype(np.float64) + A.astype(np.float64) @ W.astype(np.float64).T + bias
    scale = np.sqrt(K) * 0.05 + 1.0
    assert np.max(np.abs(host(x) - ref)) < 2e-5 * scale * 10, np.max(np.abs(host(x) - ref))


@pytest.mark.parametrize("ncand,T,d,K,frame,kv_frames,cut",
                         [(9, 258, 256, 256, 1, 3, 0),     # CTA pairs; 32-row chunks straddle
                                                           # candidates; a middle frame
                          (9, 258, 256, 256, 2, 3, 100),   # last frame, last candidate partial
                          (9, 66, 256, 128, 0, 2, 0),      # CTA pairs, blocks of 66 rows
                          (3, 40, 64, 64, 1, 2, 0)])       # single CTAs (3d = 192)
def test_linear_qkv_writes_cache_rows(planner, ncand, T, d, K, frame, kv_frames, cut):
    """QKV GEMM with the K/V-cache epilogue: q rows and the frame's cache rows hold
    bf16(A W^T + b) (within one bf16 rounding of the float64 sum), and no other cache row is
    written."""
    M = ncand * T - cut
    kv_rows = kv_frames * T
    rng = np.random.default_rng(M + d + K + frame)
    A = predictor.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = predictor.round_to_bf16((rng.standard_normal((3 * d, K)) * 0.05).astype(np.float32))
    bias = rng.standard_normal(3 * d).astype(np.float32)
    q = torch.zeros(M, d, dtype=torch.int16, device="cuda")
    kv = torch.zeros(ncand, kv_rows, 2 * d, dtype=torch.int16, device="cuda")
    planner.linear_qkv_bf16(cuda(_bf16_bits(A).astype(np.int16)), cuda(_bf16_bits(W).astype(np.int16)),
                            cuda(bias), M, d, K, T, kv_rows, frame, q, kv)
    planner.sync_check()
    ref = A.astype(np.float64) @ W.astype(np.float64).T + bias
    tol = 2.0 ** -7 * np.abs(ref) + 1e-4      # one bf16 rounding (2^-8 relative) plus slack
    got_q = _bf16_to_f64(host(q))
    assert np.all(np.abs(got_q - ref[:, :d]) <= tol[:, :d])
    kvh = host(kv)
    got_kv = _bf16_to_f64(kvh)
    rows = np.arange(M)
    c, t = rows // T, rows % T
    assert np.all(np.abs(got_kv[c, frame * T + t] - ref[:, d:]) <= tol[:, d:])
    written = np.zeros((ncand, kv_rows), bool)
    written[c, frame * T + t] = True
    assert not np.any(kvh[~written]), "cache rows outside the frame's rows were written"
