"""The C-ABI library builds, loads and exports every symbol its header declares (CPU only:
no compute call is made)."""
import ctypes
import os
import re

import pytest

from cem_search_transformer_gb300 import binding, build_lib, synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    syms = set()
    for name in os.listdir(os.path.join(ROOT, "include")):
        if name.endswith(".h"):
            text = open(os.path.join(ROOT, "include", name)).read()
            syms |= set(re.findall(r"\b(jepa_[a-z0-9_]+)\s*\(", text))
    return syms


@pytest.fixture(scope="module")
def cdll():
    path = build_lib.build()
    return ctypes.CDLL(path)


def test_every_declared_symbol_is_exported(cdll):
    declared = _declared_symbols()
    assert len(declared) >= 15
    for s in sorted(declared):
        assert hasattr(cdll, s), s
    assert declared == set(binding.EXPORTS)


def test_blob_size_matches_packer(cdll):
    lib = binding.load(build_lib.LIB)
    for pc, H in ((synthetic.TINY, 1), (synthetic.SMALL, 2), (synthetic.TINY_GATED, 1),
                  (synthetic.SMALL_GATED, 2)):
        cfg = binding.make_config(pc, H)
        weights = synthetic.make_weights(pc)
        assert lib.jepa_weight_blob_bytes(ctypes.byref(cfg)) == len(binding.pack_weights(pc, weights))


def test_invalid_configs_rejected_without_gpu(cdll):
    lib = binding.load(build_lib.LIB)
    bad = binding.make_config(synthetic.TINY, 1)
    bad.heads = 3                       # width not divisible by heads
    assert lib.jepa_weight_blob_bytes(ctypes.byref(bad)) == 0
    bf = binding.make_config(synthetic.SMALL, 1)
    bf.heads = 12                       # bf16 path needs head dim 64
    assert lib.jepa_weight_blob_bytes(ctypes.byref(bf)) == 0
    gq = binding.make_config(synthetic.SMALL_GATED, 1)
    gq.mlp = 192                        # bf16 gated needs m % 128 == 0
    assert lib.jepa_weight_blob_bytes(ctypes.byref(gq)) == 0
    gq.mlp_kind = 2                     # unknown MLP kind
    gq.mlp = 256
    assert lib.jepa_weight_blob_bytes(ctypes.byref(gq)) == 0
    h = ctypes.c_void_p()
    assert lib.jepa_create(ctypes.byref(bad), 0, ctypes.byref(h)) == 2   # JEPA_ERR_SHAPE
    assert lib.jepa_status_string(6) == b"device wait timed out"
    assert lib.jepa_last_error(None) == b""


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "cem_search_transformer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_binding_refuses_host_tensors_for_device_arguments():
    """Tensor checks run before any library call: host, wrongly typed, non-contiguous or
    short tensors never reach a kernel (needs only the library file, no GPU)."""
    import torch
    from cem_search_transformer_gb300 import binding
    B, N, P, E = 1, 2, 3, 4
    z, g, e = torch.zeros(B, N, P, E), torch.zeros(B, P, E), torch.zeros(B, N)
    with pytest.raises(binding.JepaError, match="CUDA"):
        binding.energy_l1_noalloc(z, g, B, N, P, E, e)
    with pytest.raises(binding.JepaError, match="dtype"):
        binding._arg(g.double(), "goal", "f32", B * P * E)
    with pytest.raises(binding.JepaError, match="contiguous"):
        binding._arg(torch.zeros(4, 3).t(), "x", "f32", 12, host_ok=True)
    with pytest.raises(binding.JepaError, match="elements"):
        binding._arg(g, "goal", "f32", B * P * E + 1, host_ok=True)
    with pytest.raises(binding.JepaError, match="required"):
        binding._arg(None, "goal", "f32", 1)
    assert binding._arg(None, "goal", "f32", 1, optional=True) is None
    assert binding._arg(1234, "goal", "f32", 1 << 40) == 1234       # raw address: caller's word
    assert binding._arg(g, "goal", "f32", B * P * E, host_ok=True) == g.data_ptr()


def test_kernel_entry_points_check_arguments_before_the_call():
    """The residual and QKV-cache GEMM wrappers reject bad sizes and host tensors before the
    library is called (a stand-in object without a library or context takes the Planner's
    place, so a call that got past the checks would fail differently)."""
    import torch
    from cem_search_transformer_gb300 import binding

    class Unreachable:
        def __getattr__(self, name):
            def call(*args):
                raise AssertionError(f"{name} was called although an argument was invalid")
            return call

    class NoLibrary:
        lib = Unreachable()
        h = None
        _dims = binding.Planner._dims

        def _check(self, status, what):
            raise AssertionError(f"{what} returned {status} although an argument was invalid")

    M, N, K, d, T = 64, 128, 64, 64, 16
    A = torch.zeros(M, K, dtype=torch.int16)
    W = torch.zeros(N, K, dtype=torch.int16)
    x = torch.zeros(M, N)
    with pytest.raises(binding.JepaError, match="CUDA"):
        binding.Planner.linear_resid_bf16(NoLibrary(), A, W, None, M, N, K, x)
    with pytest.raises(binding.JepaError, match=">= 1"):
        binding.Planner.linear_resid_bf16(NoLibrary(), A, W, None, 0, N, K, x)
    Wq = torch.zeros(3 * d, K, dtype=torch.int16)
    q = torch.zeros(M, d, dtype=torch.int16)
    kv = torch.zeros(M // T, 2 * T, 2 * d, dtype=torch.int16)
    with pytest.raises(binding.JepaError, match="CUDA"):
        binding.Planner.linear_qkv_bf16(NoLibrary(), A, Wq, None, M, d, K, T, 2 * T, 1, q, kv)
    with pytest.raises(binding.JepaError, match=">= 1"):
        binding.Planner.linear_qkv_bf16(NoLibrary(), A, Wq, None, M, d, K, 0, 2 * T, 1, q, kv)
