"""Attention row: block-causal attention over the KV cache (tcgen05 kernel, 128-query tiles,
the last one partial) against the oracle's attention, element-wise."""
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


def _bits(x):
    return (predictor.round_to_bf16(x).view(np.uint32) >> 16).astype(np.uint16)


def _from_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("T,Lk_blocks,heads,ncand", [(258, 1, 16, 3), (258, 3, 4, 2),
                                                      (130, 2, 2, 3), (66, 2, 6, 2),
                                                      (256, 1, 1, 1), (300, 1, 2, 1),
                                                      (129, 2, 3, 2), (387, 1, 2, 2),
                                                      (387, 2, 1, 1), (263, 1, 2, 3),
                                                      (136, 2, 3, 2),
                                                      # several items per CTA; a 1-row last
                                                      # tile; 7 key chunks
                                                      (258, 1, 16, 24), (257, 2, 2, 3),
                                                      (258, 3, 8, 30)])
def test_attention_matches_oracle(planner, T, Lk_blocks, heads, ncand):
    d = heads * 64
    kv_rows = 3 * T
    Lk = Lk_blocks * T
    rng = np.random.default_rng(T * 7 + heads)
    q = _bits(rng.standard_normal((ncand * T, d)).astype(np.float32) * 0.7)
    kv = _bits(rng.standard_normal((ncand, kv_rows, 2 * d)).astype(np.float32) * 0.7)
    out = torch.zeros(ncand * T, d, dtype=torch.int16, device="cuda")
    planner.attention_bf16(cuda(q.view(np.int16)), cuda(kv.view(np.int16)), out, ncand, T, Lk,
                           kv_rows, heads, d)
    planner.sync_check()
    got = _from_bits(host(out).view(np.uint16)).reshape(ncand, T, heads, 64)
    qf = _from_bits(q).reshape(ncand, T, heads, 64).transpose(0, 2, 1, 3).astype(np.float64)
    kf = _from_bits(kv[:, :Lk, :d]).reshape(ncand, Lk, heads, 64).transpose(0, 2, 1, 3).astype(np.float64)
    vf = _from_bits(kv[:, :Lk, d:]).reshape(ncand, Lk, heads, 64).transpose(0, 2, 1, 3).astype(np.float64)
    ref = predictor.attention(qf, kf, vf, np.ones((T, Lk), bool)).transpose(0, 2, 1, 3)
    err = np.abs(got - ref)
    # bf16 probabilities and bf16 output: a few e-3 absolute for O(0.7) values
    assert err.max() < 3e-2, err.max()
    assert err.mean() < 3e-3, err.mean()
    # the rows of the last, partial tile on their own
    tail = slice((T // 128) * 128, T)
    if T % 128:
        assert np.abs(got[:, tail] - ref[:, tail]).max() < 3e-2
