"""Pins for the oracle's candidate sampler (Philox4x32-10 + Box-Muller), CPU only."""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest

from oracle import philox

_CURAND_PHILOX4_32_10 = 161  # curandRngType_t value of CURAND_RNG_PSEUDO_PHILOX4_32_10


def _load_curand():
    paths = []
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        paths.append(os.path.join(cuda_home, sub, "libcurand.so"))
    found = ctypes.util.find_library("curand")
    if found:
        paths.append(found)
    for p in paths:
        try:
            return ctypes.CDLL(p)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def _curand_host(lib, seed, n, offset):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), _CURAND_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


@pytest.mark.parametrize("seed", [0, 42, 0x123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host_stream(seed):
    """cuRAND's host Philox4_32_10 emits block i of 4 words from counter
    (i >> 16, i >> 48, i mod 2^16, 0) with key (seed lo, seed hi): a library pin
    of the round function, the constants, the key schedule and counter words 0-2."""
    lib = _load_curand()
    k0, k1 = seed & 0xFFFFFFFF, seed >> 32
    # a contiguous run (counter word 2) ...
    out = _curand_host(lib, seed, 4 * 3000, 0).reshape(-1, 4)
    i = np.arange(3000, dtype=np.uint64)
    ref = philox.philox4x32_10(i >> np.uint64(16), i >> np.uint64(48), i & np.uint64(0xFFFF), 0, k0, k1)
    assert np.array_equal(np.stack(ref, axis=1).astype(np.uint32), out)
    # ... and offsets reaching counter words 0 and 1 (high bits of the block index)
    for blk in (2 ** 16 * 5 + 7, 2 ** 32 * 3 + 2 ** 16 * 9 + 1, 2 ** 48 * 3 + 2 ** 16 * 5 + 7,
                2 ** 60 + 2 ** 50 + 2 ** 17 + 1):
        got = _curand_host(lib, seed, 4, 4 * blk)
        ref = philox.philox4x32_10((blk >> 16) & 0xFFFFFFFF, blk >> 48, blk & 0xFFFF, 0, k0, k1)
        assert [int(v) for v in ref] == [int(v) for v in got], hex(blk)


def test_uniform_map_endpoints():
    # ((x >> 9) + 0.5) * 2^-23: smallest/largest/midpoint words
    u = philox.uniform_open01(np.array([0, 0xFFFFFFFF, 0x80000000, 511, 512], np.uint64))
    assert u[0] == 2.0 ** -24
    assert u[1] == 1.0 - 2.0 ** -24
    assert u[2] == 0.5 + 2.0 ** -24
    assert u[3] == 2.0 ** -24          # low 9 bits are discarded
    assert u[4] == 3 * 2.0 ** -24
    assert np.all((u > 0) & (u < 1))


def test_box_muller_closed_forms():
    # u0 = e^{-1/2} -> radius 1 ; u0 = e^{-2} -> radius 2 ; u0 = 1/2 -> radius sqrt(2 ln 2)
    z0, z1 = philox.box_muller(np.array([math.exp(-0.5)]), np.array([0.0]))
    assert abs(z0[0] - 1.0) < 1e-15 and abs(z1[0]) < 1e-15
    z0, z1 = philox.box_muller(np.array([math.exp(-2.0)]), np.array([0.5]))
    assert abs(z0[0] + 2.0) < 1e-15 and abs(z1[0]) < 1e-15
    z0, z1 = philox.box_muller(np.array([0.5]), np.array([0.25]))
    assert abs(z0[0]) < 1e-15 and abs(z1[0] - 1.1774100225154747) < 1e-15
    z0, z1 = philox.box_muller(np.array([0.5]), np.array([0.125]))
    assert abs(z0[0] - 0.8325546111576977) < 1e-15 and abs(z1[0] - 0.8325546111576977) < 1e-15


def test_eps_is_standard_normal():
    from scipy import stats
    eps = philox.sample_eps(42, 0, 0, 150000, 1, 7).ravel()        # ~10^6 draws
    n = eps.size
    assert abs(eps.mean()) < 5 / math.sqrt(n)
    assert abs(eps.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    assert stats.kstest(eps, "norm").pvalue > 1e-3
    # cos and sin halves of one Box-Muller pair are uncorrelated
    e = philox.sample_eps(42, 0, 0, 200000, 1, 4).reshape(-1, 4)
    assert abs(np.corrcoef(e[:, 0], e[:, 1])[0, 1]) < 0.02
    assert abs(np.corrcoef(e[:, 0], e[:, 2])[0, 1]) < 0.02


def test_eps_independent_of_batching():
    """Draws are addressed by (n, b, r): fewer candidates give a prefix (shard invariance)."""
    a = philox.sample_eps(42, 3, 5, 37, 3, 7)
    b = philox.sample_eps(42, 3, 5, 800, 3, 7)
    assert np.array_equal(a, b[:37])
    assert not np.array_equal(philox.sample_eps(42, 3, 6, 37, 3, 7), a)
    assert not np.array_equal(philox.sample_eps(42, 2, 5, 37, 3, 7), a)
    assert not np.array_equal(philox.sample_eps(43, 3, 5, 37, 3, 7), a)


def test_eps_element_to_word_mapping():
    """Element e of a candidate's H*A draws is word e % 4 of quad e // 4 (checked on raw words)."""
    seed, b, r, N, H, A = 7, 1, 2, 3, 2, 7
    Q = (H * A + 3) // 4
    eps = philox.sample_eps(seed, b, r, N, H, A).reshape(N, H * A)
    for n in range(N):
        for q in range(Q):
            w = philox.philox4x32_10(n, b, r * Q + q, 0, seed, 0)
            u = [philox.uniform_open01(v) for v in w]
            r01, r23 = math.sqrt(-2 * math.log(u[0])), math.sqrt(-2 * math.log(u[2]))
            want = [r01 * math.cos(2 * math.pi * u[1]), r01 * math.sin(2 * math.pi * u[1]),
                    r23 * math.cos(2 * math.pi * u[3]), r23 * math.sin(2 * math.pi * u[3])]
            for t in range(4):
                e = 4 * q + t
                if e < H * A:
                    assert abs(eps[n, e] - want[t]) < 1e-12


def test_sample_actions_clip_and_degenerate_sigma():
    mu = np.array([[0.5, -2.0, 0.0]])
    sig = np.zeros((1, 3))
    eps = philox.sample_eps(1, 0, 0, 5, 1, 3)
    a = philox.sample_actions(mu, sig, eps)
    assert np.array_equal(a, np.broadcast_to(np.array([[0.5, -1.0, 0.0]]), a.shape))
    a = philox.sample_actions(np.zeros((1, 3)), np.full((1, 3), 10.0), eps)
    assert a.min() >= -1.0 and a.max() <= 1.0
