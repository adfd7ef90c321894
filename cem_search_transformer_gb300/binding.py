"""Thin ctypes binding over libjepa.so (the C ABI in include/jepa_cem.h).

Argument marshalling only: every step of the planning path runs in the library's CUDA
kernels. torch is used for device memory and streams. There is no fallback: if the
library is missing or fails to load, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import struct
from typing import Dict, Optional

import numpy as np

from . import synthetic

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libjepa.so")
_lib = None

JEPA_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "shape", 3: "not loaded", 4: "out of memory",
          5: "CUDA error", 6: "timeout", 7: "unsupported"}
EXPORTS = ("jepa_create", "jepa_destroy", "jepa_last_error", "jepa_status_string",
           "jepa_weight_blob_bytes", "jepa_load_weights", "jepa_sample_actions", "jepa_philox4x32_10",
           "jepa_predictor_forward", "jepa_cem_select_refit", "jepa_cem_plan",
           "jepa_plan_kernel_count", "jepa_linear_bf16", "jepa_profile_enable",
           "jepa_profile_read", "jepa_sync_check", "jepa_energy_l1_noalloc",
           "jepa_attention_bf16", "jepa_cem_warm_start", "jepa_world_model_step",
           "jepa_cem_closed_loop", "jepa_linear_fp8", "jepa_quantize_rows_fp8",
           "jepa_set_use_graphs", "jepa_selftest_bounded_wait")


class JepaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("width", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("mlp", ctypes.c_int32), ("patch_tokens", ctypes.c_int32),
                ("embed_dim", ctypes.c_int32), ("action_dim", ctypes.c_int32),
                ("state_dim", ctypes.c_int32), ("max_horizon", ctypes.c_int32),
                ("precision", ctypes.c_int32), ("ln_eps", ctypes.c_float),
                ("max_chunk", ctypes.c_int32), ("mlp_kind", ctypes.c_int32)]

MLP_KINDS = {"gelu": 0, "gated": 1}
PRECISIONS = {"fp32": 0, "bf16": 1, "fp8": 2}


class Trace(ctypes.Structure):
    _fields_ = [("mu", ctypes.c_void_p), ("sigma", ctypes.c_void_p), ("actions", ctypes.c_void_p),
                ("energy", ctypes.c_void_p), ("elites", ctypes.c_void_p),
                ("winner", ctypes.c_void_p)]


def load(path: str = _LIB_PATH):
    """Load the library (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (__graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    sig = {
        "jepa_create": ([ctypes.POINTER(Config), I, ctypes.POINTER(P)], I),
        "jepa_destroy": ([P], None),
        "jepa_last_error": ([P], ctypes.c_char_p),
        "jepa_status_string": ([I], ctypes.c_char_p),
        "jepa_weight_blob_bytes": ([ctypes.POINTER(Config)], ctypes.c_size_t),
        "jepa_load_weights": ([P, P, ctypes.c_size_t], I),
        "jepa_sample_actions": ([P, P, P, I, I, I, I, U64, P, P], I),
        "jepa_philox4x32_10": ([P, P, U64, I, P, P], I),
        "jepa_predictor_forward": ([P, P, P, P, I, I, I, P, P, P, P], I),
        "jepa_cem_select_refit": ([P, P, P, I, I, I, I, P, P, P, P], I),
        "jepa_cem_plan": ([P, P, P, P, P, P, I, I, I, I, I, U64, P, ctypes.POINTER(Trace), P], I),
        "jepa_plan_kernel_count": ([P, I, I, I, I, I, ctypes.POINTER(ctypes.c_int64)], I),
        "jepa_linear_bf16": ([P, P, P, P, I, I, I, I, P, P], I),
        "jepa_profile_enable": ([P, I], I),
        "jepa_profile_read": ([P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_int64)], I),
        "jepa_sync_check": ([P, P], I),
        "jepa_attention_bf16": ([P, P, P, P, I, I, I, I, I, I, P], I),
        "jepa_energy_l1_noalloc": ([P, P, I, I, I, I, P, P, ctypes.c_char_p, ctypes.c_size_t], I),
        "jepa_cem_warm_start": ([P, P, P, P, I, I, P, P, P], I),
        "jepa_world_model_step": ([P, P, P, P, I, P, P, P, P, P], I),
        "jepa_cem_closed_loop": ([P, P, P, P, P, P, I, I, I, I, I, I, I, U64, P, P, P], I),
        "jepa_linear_fp8": ([P, P, P, P, P, P, I, I, I, I, P, P], I),
        "jepa_quantize_rows_fp8": ([P, P, I, I, P, P, P], I),
        "jepa_set_use_graphs": ([P, I], I),
        "jepa_selftest_bounded_wait": ([P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def make_config(pc: synthetic.PredictorConfig, max_horizon: int = 1, max_chunk: int = 0) -> Config:
    return Config(pc.layers, pc.width, pc.heads, pc.mlp, pc.patch_tokens, pc.embed_dim,
                  pc.action_dim, pc.state_dim, max_horizon, PRECISIONS[pc.precision],
                  pc.ln_eps, max_chunk, MLP_KINDS[pc.mlp_kind])


def pack_weights(pc: synthetic.PredictorConfig, weights: Dict[str, np.ndarray]) -> bytes:
    """Weight blob: 64-byte header + fp32 tensors in canonical order (format only)."""
    hdr = struct.pack("<11i", 0x4150454A, 1, pc.layers, pc.width, pc.heads, pc.mlp,
                      pc.patch_tokens, pc.embed_dim, pc.action_dim, pc.state_dim,
                      MLP_KINDS[pc.mlp_kind]).ljust(64, b"\0")
    shapes = synthetic.weight_shapes(pc)
    parts = [hdr]
    for name in synthetic.weight_names(pc):
        w = np.ascontiguousarray(weights[name], dtype=np.float32)
        assert w.shape == shapes[name], (name, w.shape)
        parts.append(w.tobytes())
    return b"".join(parts)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def energy_l1_noalloc(z_pred, goal, B, N, P, E, energy, stream=None):
    """L1 energy of predicted frames without any device allocation (see the C header).

    For callers that cannot allocate device memory (a fixed memory budget owned by a host
    framework, or a control loop that must not allocate mid-episode). Raises JepaError with
    the library's message on failure, e.g. when B*N*ceil(P/32) exceeds the fixed scratch."""
    lib = load()
    buf = ctypes.create_string_buffer(256)
    st = lib.jepa_energy_l1_noalloc(_ptr(z_pred), _ptr(goal), B, N, P, E, _ptr(energy),
                                    _stream(stream), buf, len(buf))
    if st != JEPA_OK:
        raise JepaError(st, buf.value.decode())


class Planner:
    """One library context (weights + workspaces + captured graphs) on one device."""

    def __init__(self, pc: synthetic.PredictorConfig, max_horizon: int = 1, device: int = 0,
                 max_chunk: int = 0):
        self.lib = load()
        self.pc = pc
        self.cfg = make_config(pc, max_horizon, max_chunk)
        h = ctypes.c_void_p()
        st = self.lib.jepa_create(ctypes.byref(self.cfg), device, ctypes.byref(h))
        if st != JEPA_OK:
            raise JepaError(st, "jepa_create")
        self.h = h

    def _check(self, st: int, what: str):
        if st != JEPA_OK:
            raise JepaError(st, f"{what}: {self.lib.jepa_last_error(self.h).decode()}")

    def close(self):
        if getattr(self, "h", None):
            self.lib.jepa_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def blob_bytes(self) -> int:
        return self.lib.jepa_weight_blob_bytes(ctypes.byref(self.cfg))

    def load_weights(self, weights: Dict[str, np.ndarray]):
        blob = pack_weights(self.pc, weights)
        buf = ctypes.create_string_buffer(blob, len(blob))
        self._check(self.lib.jepa_load_weights(self.h, buf, len(blob)), "load_weights")

    def load_blob(self, blob: bytes):
        buf = ctypes.create_string_buffer(blob, len(blob))
        return self.lib.jepa_load_weights(self.h, buf, len(blob))

    def sample_actions(self, mu, sigma, B, N, H, rnd, seed, actions, stream=None):
        self._check(self.lib.jepa_sample_actions(self.h, _ptr(mu), _ptr(sigma), B, N, H, rnd, seed,
                                                 _ptr(actions), _stream(stream)), "sample_actions")

    def philox(self, counters, seed, n, out, stream=None):
        self._check(self.lib.jepa_philox4x32_10(self.h, _ptr(counters), seed, n, _ptr(out),
                                                _stream(stream)), "philox4x32_10")

    def predictor_forward(self, z_ctx, state0, actions, B, N, H, goal=None, z_pred=None,
                          energy=None, stream=None):
        self._check(self.lib.jepa_predictor_forward(
            self.h, _ptr(z_ctx), _ptr(state0), _ptr(actions), B, N, H, _ptr(goal), _ptr(z_pred),
            _ptr(energy), _stream(stream)), "predictor_forward")

    def select_refit(self, energy, actions, B, N, H, K, mu_out, sigma_out, elites_out=None,
                     stream=None):
        self._check(self.lib.jepa_cem_select_refit(
            self.h, _ptr(energy), _ptr(actions), B, N, H, K, _ptr(mu_out), _ptr(sigma_out),
            _ptr(elites_out), _stream(stream)), "select_refit")

    def plan(self, z0, state0, goal, mu0, sigma0, B, H, N, K, rounds, seed, action_out,
             trace: Optional[Dict[str, object]] = None, stream=None):
        """Inputs/outputs may be torch CUDA tensors, or raw host/device addresses (int)."""
        tr = None
        if trace is not None:
            tr = Trace(*(_ptr(trace.get(k)) for k in ("mu", "sigma", "actions", "energy",
                                                         "elites", "winner")))
        self._check(self.lib.jepa_cem_plan(
            self.h, _ptr(z0), _ptr(state0), _ptr(goal), _ptr(mu0), _ptr(sigma0), B, H, N, K,
            rounds, seed, _ptr(action_out), ctypes.byref(tr) if tr is not None else None,
            _stream(stream)), "cem_plan")

    def warm_start(self, mu_prev, mu_prior, sigma_prior, B, H, mu_out, sigma_out, stream=None):
        self._check(self.lib.jepa_cem_warm_start(
            self.h, _ptr(mu_prev), _ptr(mu_prior), _ptr(sigma_prior), B, H, _ptr(mu_out),
            _ptr(sigma_out), _stream(stream)), "cem_warm_start")

    def world_model_step(self, z, state, action, B, z_next, state_next, goal=None, distance=None,
                         stream=None):
        self._check(self.lib.jepa_world_model_step(
            self.h, _ptr(z), _ptr(state), _ptr(action), B, _ptr(goal), _ptr(z_next),
            _ptr(state_next), _ptr(distance), _stream(stream)), "world_model_step")

    def closed_loop(self, z0, state0, goal, mu_prior, sigma_prior, B, H, N, K, rounds, steps,
                    warm, seed, actions_out, distance_out, stream=None):
        self._check(self.lib.jepa_cem_closed_loop(
            self.h, _ptr(z0), _ptr(state0), _ptr(goal), _ptr(mu_prior), _ptr(sigma_prior), B, H,
            N, K, rounds, steps, int(warm), seed, _ptr(actions_out), _ptr(distance_out),
            _stream(stream)), "cem_closed_loop")

    def kernel_count(self, B, H, N, K, rounds) -> int:
        c = ctypes.c_int64()
        self._check(self.lib.jepa_plan_kernel_count(self.h, B, H, N, K, rounds, ctypes.byref(c)),
                    "plan_kernel_count")
        return c.value

    def linear_bf16(self, A, W, bias, M, N, K, gelu, out, stream=None):
        self._check(self.lib.jepa_linear_bf16(self.h, _ptr(A), _ptr(W), _ptr(bias), M, N, K,
                                              int(gelu), _ptr(out), _stream(stream)), "linear_bf16")

    def linear_fp8(self, A, a_scale, W, w_scale, bias, M, N, K, gelu, out, stream=None):
        self._check(self.lib.jepa_linear_fp8(self.h, _ptr(A), _ptr(a_scale), _ptr(W), _ptr(w_scale),
                                             _ptr(bias), M, N, K, int(gelu), _ptr(out),
                                             _stream(stream)), "linear_fp8")

    def quantize_rows_fp8(self, x, rows, cols, codes, scales, stream=None):
        self._check(self.lib.jepa_quantize_rows_fp8(self.h, _ptr(x), rows, cols, _ptr(codes),
                                                    _ptr(scales), _stream(stream)),
                    "quantize_rows_fp8")

    def attention_bf16(self, q, kv, out, ncand, T, Lk, kv_rows, heads, d, stream=None):
        self._check(self.lib.jepa_attention_bf16(self.h, _ptr(q), _ptr(kv), _ptr(out), ncand, T, Lk,
                                                 kv_rows, heads, d, _stream(stream)),
                    "attention_bf16")

    def set_use_graphs(self, on: bool):
        self._check(self.lib.jepa_set_use_graphs(self.h, int(on)), "set_use_graphs")

    def profile_enable(self, on: bool):
        self._check(self.lib.jepa_profile_enable(self.h, int(on)), "profile_enable")

    def profile_read(self):
        ms, fl, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int64()
        self._check(self.lib.jepa_profile_read(self.h, ctypes.byref(ms), ctypes.byref(fl),
                                               ctypes.byref(n)), "profile_read")
        return ms.value, fl.value, n.value

    def selftest_bounded_wait(self, stream=None):
        self._check(self.lib.jepa_selftest_bounded_wait(self.h, _stream(stream)),
                    "selftest_bounded_wait")

    def sync_check(self, stream=None):
        self._check(self.lib.jepa_sync_check(self.h, _stream(stream)), "sync_check")
