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
           "jepa_set_use_graphs", "jepa_selftest_bounded_wait", "jepa_linear_resid_bf16",
           "jepa_linear_qkv_bf16")


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
        "jepa_linear_resid_bf16": ([P, P, P, P, I, I, I, P, P], I),
        "jepa_linear_qkv_bf16": ([P, P, P, P, I, I, I, I, I, I, P, P, P], I),
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


_DTYPES = {"f32": ("float32",), "bf16": ("bfloat16", "int16", "uint16"), "u8": ("uint8", "float8_e4m3fn"),
           "i32": ("int32",), "u32": ("int32", "uint32")}


def _arg(t, name: str, kind: str, numel: int, host_ok: bool = False,
         optional: bool = False) -> Optional[int]:
    """Address of argument `t` after checking that it can hold `numel` elements of `kind`.

    A torch tensor must have that element type, be contiguous, hold at least `numel`
    elements and live on a CUDA device (or, where `host_ok`, in host memory); anything else
    raises JepaError(INVALID_ARG) before the library is called, so that no kernel reads or
    writes past a caller's buffer. A raw integer address is passed through unchecked: the
    caller vouches for its size and location. None is allowed only for optional arguments."""
    if t is None:
        if optional:
            return None
        raise JepaError(1, f"{name} is required")
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise JepaError(1, f"{name}: expected a torch tensor or an integer address, got {type(t).__name__}")
    if str(t.dtype).replace("torch.", "") not in _DTYPES[kind]:
        raise JepaError(1, f"{name}: dtype {t.dtype} where {kind} is required")
    if not t.is_contiguous():
        raise JepaError(1, f"{name} must be contiguous")
    if not t.is_cuda and not host_ok:
        raise JepaError(1, f"{name} must be a CUDA tensor")
    if t.numel() < numel:
        raise JepaError(1, f"{name} holds {t.numel()} elements, {numel} are needed")
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
    if min(B, N, P, E) < 1:
        raise JepaError(1, "energy_l1_noalloc: B, N, P and E must be positive")
    zp = _arg(z_pred, "z_pred", "f32", B * N * P * E)
    gp = _arg(goal, "goal", "f32", B * P * E)
    ep = _arg(energy, "energy", "f32", B * N)
    buf = ctypes.create_string_buffer(256)
    st = lib.jepa_energy_l1_noalloc(zp, gp, B, N, P, E, ep, _stream(stream), buf, len(buf))
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

    def _dims(self, **sizes):
        for k, v in sizes.items():
            if int(v) < 1:
                raise JepaError(1, f"{k} must be >= 1 (got {v})")

    def sample_actions(self, mu, sigma, B, N, H, rnd, seed, actions, stream=None):
        self._dims(B=B, N=N, H=H)
        A = self.pc.action_dim
        self._check(self.lib.jepa_sample_actions(
            self.h, _arg(mu, "mu", "f32", B * H * A), _arg(sigma, "sigma", "f32", B * H * A), B, N,
            H, rnd, seed, _arg(actions, "actions", "f32", B * N * H * A), _stream(stream)),
            "sample_actions")

    def philox(self, counters, seed, n, out, stream=None):
        self._dims(n=n)
        self._check(self.lib.jepa_philox4x32_10(self.h, _arg(counters, "counters", "u32", 4 * n),
                                                seed, n, _arg(out, "out", "u32", 4 * n),
                                                _stream(stream)), "philox4x32_10")

    def predictor_forward(self, z_ctx, state0, actions, B, N, H, goal=None, z_pred=None,
                          energy=None, stream=None):
        self._dims(B=B, N=N, H=H)
        pc, PE = self.pc, self.pc.patch_tokens * self.pc.embed_dim
        self._check(self.lib.jepa_predictor_forward(
            self.h, _arg(z_ctx, "z_ctx", "f32", B * PE), _arg(state0, "state0", "f32", B * pc.state_dim),
            _arg(actions, "actions", "f32", B * N * H * pc.action_dim), B, N, H,
            _arg(goal, "goal", "f32", B * PE, optional=True),
            _arg(z_pred, "z_pred", "f32", B * N * PE, optional=True),
            _arg(energy, "energy", "f32", B * N, optional=True), _stream(stream)), "predictor_forward")

    def select_refit(self, energy, actions, B, N, H, K, mu_out, sigma_out, elites_out=None,
                     stream=None):
        self._dims(B=B, N=N, H=H, K=K)
        HA = H * self.pc.action_dim
        self._check(self.lib.jepa_cem_select_refit(
            self.h, _arg(energy, "energy", "f32", B * N), _arg(actions, "actions", "f32", B * N * HA),
            B, N, H, K, _arg(mu_out, "mu_out", "f32", B * HA), _arg(sigma_out, "sigma_out", "f32", B * HA),
            _arg(elites_out, "elites_out", "i32", B * K, optional=True), _stream(stream)),
            "select_refit")

    def plan(self, z0, state0, goal, mu0, sigma0, B, H, N, K, rounds, seed, action_out,
             trace: Optional[Dict[str, object]] = None, stream=None):
        """Inputs and action_out may be torch tensors (CUDA or host) or raw host/device
        addresses (int); the trace's buffers are CUDA tensors or device addresses."""
        self._dims(B=B, H=H, N=N, K=K, rounds=rounds)
        pc = self.pc
        PE, HA, R = pc.patch_tokens * pc.embed_dim, H * pc.action_dim, rounds
        tr = None
        if trace is not None:
            sizes = {"mu": ("f32", (R + 1) * B * HA), "sigma": ("f32", (R + 1) * B * HA),
                     "actions": ("f32", R * B * N * HA), "energy": ("f32", R * B * N),
                     "elites": ("i32", R * B * K), "winner": ("i32", B)}
            tr = Trace(*(_arg(trace.get(k), f"trace[{k}]", sizes[k][0], sizes[k][1], optional=True)
                         for k in ("mu", "sigma", "actions", "energy", "elites", "winner")))
        self._check(self.lib.jepa_cem_plan(
            self.h, _arg(z0, "z0", "f32", B * PE, host_ok=True),
            _arg(state0, "state0", "f32", B * pc.state_dim, host_ok=True),
            _arg(goal, "goal", "f32", B * PE, host_ok=True),
            _arg(mu0, "mu0", "f32", B * HA, host_ok=True),
            _arg(sigma0, "sigma0", "f32", B * HA, host_ok=True), B, H, N, K, rounds, seed,
            _arg(action_out, "action_out", "f32", B * pc.action_dim, host_ok=True),
            ctypes.byref(tr) if tr is not None else None, _stream(stream)), "cem_plan")

    def warm_start(self, mu_prev, mu_prior, sigma_prior, B, H, mu_out, sigma_out, stream=None):
        self._dims(B=B, H=H)
        n = B * H * self.pc.action_dim
        self._check(self.lib.jepa_cem_warm_start(
            self.h, _arg(mu_prev, "mu_prev", "f32", n), _arg(mu_prior, "mu_prior", "f32", n),
            _arg(sigma_prior, "sigma_prior", "f32", n), B, H, _arg(mu_out, "mu_out", "f32", n),
            _arg(sigma_out, "sigma_out", "f32", n), _stream(stream)), "cem_warm_start")

    def world_model_step(self, z, state, action, B, z_next, state_next, goal=None, distance=None,
                         stream=None):
        self._dims(B=B)
        pc, PE = self.pc, self.pc.patch_tokens * self.pc.embed_dim
        self._check(self.lib.jepa_world_model_step(
            self.h, _arg(z, "z", "f32", B * PE), _arg(state, "state", "f32", B * pc.state_dim),
            _arg(action, "action", "f32", B * pc.action_dim), B,
            _arg(goal, "goal", "f32", B * PE, optional=True), _arg(z_next, "z_next", "f32", B * PE),
            _arg(state_next, "state_next", "f32", B * pc.state_dim),
            _arg(distance, "distance", "f32", B, optional=True), _stream(stream)), "world_model_step")

    def closed_loop(self, z0, state0, goal, mu_prior, sigma_prior, B, H, N, K, rounds, steps,
                    warm, seed, actions_out, distance_out, stream=None):
        self._dims(B=B, H=H, N=N, K=K, rounds=rounds, steps=steps)
        pc = self.pc
        PE, HA = pc.patch_tokens * pc.embed_dim, H * pc.action_dim
        self._check(self.lib.jepa_cem_closed_loop(
            self.h, _arg(z0, "z0", "f32", B * PE, host_ok=True),
            _arg(state0, "state0", "f32", B * pc.state_dim, host_ok=True),
            _arg(goal, "goal", "f32", B * PE, host_ok=True),
            _arg(mu_prior, "mu_prior", "f32", B * HA, host_ok=True),
            _arg(sigma_prior, "sigma_prior", "f32", B * HA, host_ok=True), B, H, N, K, rounds, steps,
            int(warm), seed, _arg(actions_out, "actions_out", "f32", steps * B * pc.action_dim,
                                  host_ok=True),
            _arg(distance_out, "distance_out", "f32", steps * B, host_ok=True), _stream(stream)),
            "cem_closed_loop")

    def kernel_count(self, B, H, N, K, rounds) -> int:
        c = ctypes.c_int64()
        self._check(self.lib.jepa_plan_kernel_count(self.h, B, H, N, K, rounds, ctypes.byref(c)),
                    "plan_kernel_count")
        return c.value

    def linear_bf16(self, A, W, bias, M, N, K, gelu, out, stream=None):
        self._dims(M=M, N=N, K=K)
        n_out = N // 2 if int(gelu) == 2 else N
        self._check(self.lib.jepa_linear_bf16(
            self.h, _arg(A, "A", "bf16", M * K), _arg(W, "W", "bf16", N * K),
            _arg(bias, "bias", "f32", N, optional=True), M, N, K, int(gelu),
            _arg(out, "out", "f32", M * n_out), _stream(stream)), "linear_bf16")

    def linear_resid_bf16(self, A, W, bias, M, N, K, x, stream=None):
        self._dims(M=M, N=N, K=K)
        self._check(self.lib.jepa_linear_resid_bf16(
            self.h, _arg(A, "A", "bf16", M * K), _arg(W, "W", "bf16", N * K),
            _arg(bias, "bias", "f32", N, optional=True), M, N, K,
            _arg(x, "x", "f32", M * N), _stream(stream)), "linear_resid_bf16")

    def linear_qkv_bf16(self, A, W, bias, M, d, K, T, kv_rows, frame, q, kv, stream=None):
        self._dims(M=M, d=d, K=K, T=T, kv_rows=kv_rows)
        ncand = -(-int(M) // int(T))
        self._check(self.lib.jepa_linear_qkv_bf16(
            self.h, _arg(A, "A", "bf16", M * K), _arg(W, "W", "bf16", 3 * d * K),
            _arg(bias, "bias", "f32", 3 * d, optional=True), M, d, K, T, kv_rows, int(frame),
            _arg(q, "q", "bf16", M * d), _arg(kv, "kv", "bf16", ncand * kv_rows * 2 * d),
            _stream(stream)), "linear_qkv_bf16")

    def linear_fp8(self, A, a_scale, W, w_scale, bias, M, N, K, gelu, out, stream=None):
        self._dims(M=M, N=N, K=K)
        n_out = N // 2 if int(gelu) == 2 else N
        self._check(self.lib.jepa_linear_fp8(
            self.h, _arg(A, "A", "u8", M * K), _arg(a_scale, "a_scale", "f32", M),
            _arg(W, "W", "u8", N * K), _arg(w_scale, "w_scale", "f32", N),
            _arg(bias, "bias", "f32", N, optional=True), M, N, K, int(gelu),
            _arg(out, "out", "f32", M * n_out), _stream(stream)), "linear_fp8")

    def quantize_rows_fp8(self, x, rows, cols, codes, scales, stream=None):
        self._dims(rows=rows, cols=cols)
        self._check(self.lib.jepa_quantize_rows_fp8(
            self.h, _arg(x, "x", "f32", rows * cols), rows, cols,
            _arg(codes, "codes", "u8", rows * cols), _arg(scales, "scales", "f32", rows),
            _stream(stream)), "quantize_rows_fp8")

    def attention_bf16(self, q, kv, out, ncand, T, Lk, kv_rows, heads, d, stream=None):
        self._dims(ncand=ncand, T=T, Lk=Lk, kv_rows=kv_rows, heads=heads, d=d)
        self._check(self.lib.jepa_attention_bf16(
            self.h, _arg(q, "q", "bf16", ncand * T * d), _arg(kv, "kv", "bf16", ncand * kv_rows * 2 * d),
            _arg(out, "out", "bf16", ncand * T * d), ncand, T, Lk, kv_rows, heads, d,
            _stream(stream)), "attention_bf16")

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
