"""Benchmark: one CEM planning step over the full-shape action-conditioned predictor.

Workload (default "full"): 24-layer, width-1024, 16-head, MLP-4096 predictor with 256 patch
tokens of dim 1408 plus action and state tokens; N=800 candidates, K=80 elites, R=10
rounds, horizon 1; seeded random weights N(0, 0.02) and N(0, 1) embeddings. A step is one
full planning step (all rounds, through jepa_cem_plan). The metric is candidate rollouts per
second (N * R * B / step time); ms per step is reported beside it.

  python bench.py [--gpus N --steps K --warmup W --workload NAME --impl ours|reference]
  python bench.py --closed-loop T [--rounds R] [--warm] [--workload NAME]

The --closed-loop mode times a receding-horizon episode instead ("Further Optimization",
parts A and B of the planning page): T control steps, each a full plan followed by one
world-model step that executes the winner's first action, optionally warm-started from
the previous plan; it prints one JSON line with ms per control step and the L1 distance
to the goal after every step.

Under torchrun (N > 1) each rank plans its own independent problem (weak scaling, no
collective on the data path); rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from cem_search_transformer_gb300 import synthetic  # noqa: E402

METRIC = "CEM plan-step latency (ms, 800x10) and candidate rollouts/sec, % of roofline"
# DRAM bytes (read + write) per launch of the four per-layer GEMMs (QKV, out-projection,
# MLP up, MLP down) on the full-shape workload: one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of 512 candidates (132,096 rows, operands above the L2), scaled by
# 800 / 512 to the 206,400 rows of a full launch (the traffic is proportional to the rows;
# the weights are a few MB). Taken from the GEMM kernels whose source hashes to
# GEMM_TRAFFIC_SOURCE_SHA (first 16 hex digits of the SHA-256 of gemm_tc.cu, tc_common.cuh
# and common.cuh, in that order); when the kernels change, the line reports no traffic until
# the counters are taken again.
GEMM_DRAM_BYTES_PER_LAUNCH_FULL = (432.9e6 + 1195.3e6, 1274.0e6 + 757.2e6, 437.7e6 + 1615.8e6,
                                   2705.9e6 + 802.7e6)
GEMM_TRAFFIC_SOURCE_SHA = "f46d6499d7959abf"
PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAK_FALLBACK, "fallback"


def gemm_source_sha() -> str:
    """Hash of the GEMM kernels' source (see GEMM_TRAFFIC_SOURCE_SHA)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "cem_search_transformer_gb300", "csrc")
    for name in ("gemm_tc.cu", "tc_common.cuh", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def rank_problems(pc, B, rank):
    """Weak scaling by independent problems: rank r plans problems r*B .. r*B + B - 1 (the
    same seeded inputs a single process would draw for them)."""
    return synthetic.make_problems(pc, B, seed_base=1000 + rank * B)


def reduce_max(x: float, world: int, device) -> float:
    """Max over ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def fp8_flop_split(pc, H):
    """GEMM FLOPs per candidate rollout on e4m3 operands (QKV, MLP up, projection to E) and
    on bf16 operands (out-projection, MLP down, in-projection of predicted frames)."""
    T, P, E, d, m, L = pc.tokens, pc.patch_tokens, pc.embed_dim, pc.width, pc.mlp, pc.layers
    up = 2 * m if pc.mlp_kind == "gated" else m
    f8 = H * (L * (2 * T * 3 * d * d + 2 * T * up * d) + 2 * P * E * d)
    f16 = H * L * (2 * T * d * d + 2 * T * d * m) + (H - 1) * 2 * P * d * E
    return float(f8), float(f16)


def attention_flops(pc, H):
    """Attention FLOPs per candidate rollout: per frame k, every layer and head takes T queries
    over the (k + 1) T cached keys, Q K^T and P V at 2 FLOPs per multiply-add each."""
    T, d, L = pc.tokens, pc.width, pc.layers
    return float(sum(L * 4 * T * (k + 1) * T * d for k in range(H)))


def step_roofline(pc, H, rollouts, gemm_tflop, step_ms, peaks):
    """The whole plan step against the tensor-core roofline: executed GEMM FLOPs (measured
    count if available) plus attention FLOPs, at the measured burst and sustained bf16 rates
    and at the nominal 2.25 PFLOP/s dense bf16 of a GB300 (e4m3 GEMMs count at twice the
    bf16 rate). The operand bytes (0.61 GB of weights per pass) are far below the FLOP time."""
    f8, f16 = fp8_flop_split(pc, H)
    if pc.precision != "fp8":
        f8, f16 = 0.0, f8 + f16
    gemm = f8 + f16
    scale = (gemm_tflop * 1e12 / rollouts) / gemm if gemm_tflop else 1.0
    f8, f16 = f8 * scale * rollouts, (f16 * scale + attention_flops(pc, H)) * rollouts
    out = {"bound": "tensor", "tflop_per_step": (f8 + f16) / 1e12}
    for key, tf in (("measured_burst", peaks.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"])),
                    ("measured_sustained", peaks.get("bf16_tflops_sustained",
                                                     PEAK_FALLBACK["bf16_tflops_sustained"])),
                    ("nominal_dense", 2250.0)):
        t_ms = (f8 / (2 * tf) + f16 / tf) / 1e12 * 1e3
        out[f"ms_at_{key}"] = t_ms
        out[f"frac_of_{key}"] = t_ms / step_ms
    return out


def workload_desc(wl):
    pc = wl.predictor
    return (f"{wl.predictor.name} CEM: {pc.layers}x{pc.width} predictor, heads {pc.heads}, "
            f"MLP {pc.mlp}, P={pc.patch_tokens} E={pc.embed_dim}, N={wl.N} K={wl.K} "
            f"R={wl.rounds} H={wl.horizon} B={wl.B}")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str = ""):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(log_dir or tempfile.gettempdir(), f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


_ORACLE_WEIGHTS = {}


def _oracle_weights(pc):
    from oracle import predictor
    if pc.name not in _ORACLE_WEIGHTS:   # prepared once per process (outside every timing)
        _ORACLE_WEIGHTS[pc.name] = predictor.prepare_weights(synthetic.make_weights(pc, seed=0),
                                                             pc.precision)
    return _ORACLE_WEIGHTS[pc.name]


def _oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        return os.cpu_count()


class OracleSample:
    """Round 0's candidates of a workload, rolled out and scored by the CPU oracle (numpy
    float64): the bounded sample both CPU legs time."""

    def __init__(self, wl, problem_seed: int = 1000):
        from oracle import philox
        self.wl, self.pc = wl, wl.predictor
        self.w = _oracle_weights(self.pc)
        self.z0, self.goal, self.s0 = synthetic.make_problems(self.pc, 1, seed_base=problem_seed)
        mu0, sg0 = synthetic.make_gaussian(self.pc, 1, wl.horizon)
        self.acts = philox.sample_actions(mu0[0], sg0[0],
                                          philox.sample_eps(wl.seed, 0, 0, wl.N, wl.horizon, 7))
        self.next = 0

    def run(self, n: int) -> int:
        """Rolls out and scores the next n candidates (in batches of at most 8, wrapping
        round); returns n."""
        from oracle import predictor
        done = 0
        while done < n:
            m = min(8, n - done, self.wl.N - self.next)
            a = self.acts[self.next:self.next + m]
            predictor.energy_l1(predictor.rollout(self.w, self.pc, self.z0[0], self.s0[0], a)[-1],
                                self.goal[0])
            self.next = (self.next + m) % self.wl.N
            done += m
        return n

    def seconds_per_rollout(self) -> float:
        t0 = time.perf_counter()
        self.run(1)
        return time.perf_counter() - t0

    def describe(self, n) -> str:
        return (f"{n} candidate rollouts of round 0 (plus the select/refit, negligible) of "
                f"{workload_desc(self.wl)}; numpy float64 oracle")


def cpu_baseline(wl, budget_s: float = 15.0, problem_seed: int = 1000):
    """The CPU oracle (numpy float64) on a bounded sample of the same workload: the first
    round's candidates, as many as fit in about budget_s seconds. Returns (rollouts/s, info)."""
    smp = OracleSample(wl, problem_seed)
    t1 = smp.seconds_per_rollout()
    n = int(max(1, min(wl.N, budget_s / max(t1, 1e-6))))
    t0 = time.perf_counter()
    smp.run(n)
    dt = time.perf_counter() - t0
    return n / dt, {"cores": _oracle_cores(), "sample": smp.describe(n), "seconds": dt}


def cpu_full_configs(names=("tiny", "small")):
    """Whole planning steps of the small configurations on the host cores (oracle cem.plan,
    every candidate of every round): ms per step and candidate rollouts/s."""
    from oracle import cem
    out = {}
    for name in names:
        wl = synthetic.WORKLOADS[name]
        pc = wl.predictor
        w = synthetic.make_weights(pc, seed=0)
        z0, goal, s0 = synthetic.make_problems(pc, 1)
        mu0, sg0 = synthetic.make_gaussian(pc, 1, wl.horizon)
        t0 = time.perf_counter()
        cem.plan(w, pc, z0[0], s0[0], goal[0], mu0[0], sg0[0], wl.N, wl.K, wl.rounds, wl.seed)
        dt = time.perf_counter() - t0
        out[name] = {"ms_per_step": dt * 1e3, "rollouts_per_s": wl.N * wl.rounds / dt,
                     "workload": workload_desc(wl)}
    return out


def run_reference(args, wl):
    """The oracle as the reference arm: every step rolls out and scores a bounded sample of
    the workload's round-0 candidates on the host cores; the warm-up steps take one
    candidate each. The timed steps share a budget of --cpu-budget seconds."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    smp = OracleSample(wl)
    t1 = min(smp.seconds_per_rollout() for _ in range(max(1, args.warmup)))
    n_step = int(max(1, min(wl.N, args.cpu_budget / max(1, args.steps) / max(t1, 1e-6))))
    step_s = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        smp.run(n_step)
        step_s.append(time.perf_counter() - t0)
    value = n_step * args.steps / sum(step_s)
    sample = smp.describe(n_step) + " per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "candidate rollouts/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": float(np.mean(step_s)) * 1e3,
            "ms_per_full_step_extrapolated": wl.N * wl.rounds * wl.B / value * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) embeddings)",
            "config": {"workload": workload_desc(wl), "per_rank_problems": wl.B,
                       "parallelism": "none (host cores)",
                       "step": f"a bounded sample: {n_step} of the step's {wl.N * wl.rounds * wl.B} "
                               "candidate rollouts (ms_per_step is the sample's time)"},
            "cpu_baseline": {"value": value, "unit": "candidate rollouts/s", "cores": _oracle_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "candidate rollouts/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    from cem_search_transformer_gb300 import binding, build_lib

    rank, world, local = rank_info()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_lib.build()
    pc = wl.predictor
    B, N, K, R, H = wl.B, wl.N, wl.K, wl.rounds, wl.horizon
    planner = binding.Planner(pc, max_horizon=H, device=local)
    planner.load_weights(synthetic.make_weights(pc, seed=0))
    # each rank plans its own problems (independent units, weak scaling)
    z0, goal, s0 = rank_problems(pc, B, rank)
    mu0, sg0 = synthetic.make_gaussian(pc, B, H)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    dz0, dgoal, ds0, dmu, dsg = t(z0), t(goal), t(s0), t(mu0), t(sg0)
    out = torch.zeros(B, pc.action_dim, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, world, dev)

    if args.no_graph:
        planner.set_use_graphs(False)     # launch the graph's kernels one by one
    for _ in range(args.warmup):
        planner.plan(dz0, ds0, dgoal, dmu, dsg, B, H, N, K, R, wl.seed, out, stream=stream)
    planner.sync_check(stream)
    launches_per_step = planner.kernel_count(B, H, N, K, R)

    # ---- device-resident timing (inputs already in HBM), plain graph replay ----
    barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, args.clocks_dir) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            planner.plan(dz0, ds0, dgoal, dmu, dsg, B, H, N, K, R, wl.seed, out, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    planner.sync_check(stream)
    step_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    clocks = clk.summary()

    # ---- per-GEMM timing: a separately captured graph with event pairs around every GEMM
    # (kept out of the timed region above: the event nodes add launch gaps) ----
    gemm_ms = gemm_flops = 0.0
    gemm_launches = 0
    prof_steps = min(args.steps, 3)
    if not args.no_graph:
        planner.profile_enable(True)
        planner.plan(dz0, ds0, dgoal, dmu, dsg, B, H, N, K, R, wl.seed, out, stream=stream)
        stream.synchronize()
        for _ in range(prof_steps):
            planner.plan(dz0, ds0, dgoal, dmu, dsg, B, H, N, K, R, wl.seed, out, stream=stream)
            stream.synchronize()
            ms, fl, n = planner.profile_read()
            gemm_ms += ms
            gemm_flops += fl
            gemm_launches += n
        planner.profile_enable(False)
        planner.sync_check(stream)

    # ---- end to end through the C ABI with pinned host buffers ----
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hz0, hgoal, hs0, hmu, hsg = pin(z0), pin(goal), pin(s0), pin(mu0), pin(sg0)
    hout = torch.zeros(B, pc.action_dim).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hz0, hgoal, hs0, hmu, hsg))
    d2h = hout.numel() * hout.element_size()
    planner.plan(hz0.data_ptr(), hs0.data_ptr(), hgoal.data_ptr(), hmu.data_ptr(), hsg.data_ptr(),
                 B, H, N, K, R, wl.seed, hout.data_ptr(), stream=stream)
    stream.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        planner.plan(hz0.data_ptr(), hs0.data_ptr(), hgoal.data_ptr(), hmu.data_ptr(), hsg.data_ptr(),
                     B, H, N, K, R, wl.seed, hout.data_ptr(), stream=stream)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    planner.sync_check(stream)

    rollouts = N * R * B * world
    if rank == 0:
        peaks, peak_kind = load_peaks()
        peak = peaks.get("bf16_tflops_sustained", PEAK_FALLBACK["bf16_tflops_sustained"])
        peak_source = f"{peak_kind} bf16_tflops_sustained (kernel timed inside a long step)"
        dtype = "bf16"
        if pc.precision == "fp8":
            # e4m3 GEMMs at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense): the peak
            # for this FLOP mix is the harmonic combination of the two
            f8, f16 = fp8_flop_split(pc, H)
            peak = (f8 + f16) / (f8 / (2 * peak) + f16 / peak)
            peak_source += f"; fp8 share {f8 / (f8 + f16):.3f} of the GEMM FLOPs at 2x"
            dtype = "e4m3+bf16"
        achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
        step_flops = None
        if gemm_launches:
            step_flops = gemm_flops / prof_steps
        line = {
            "metric": METRIC, "value": rollouts / (step_ms * 1e-3), "unit": "candidate rollouts/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) embeddings)",
            "config": {"workload": workload_desc(wl), "per_rank_problems": B,
                       "parallelism": f"independent problems x{world} (no collective)",
                       "l2": "not flushed: working set (0.61 GB bf16 weights + ~4 GB activations "
                             "per round) exceeds the 129 MB L2",
                       "timing": "CUDA events on the launch stream; host sync per step",
                       "launch": "kernels launched one by one on the stream" if args.no_graph
                                 else "one CUDA graph replay per step"},
            "roofline": {"bound": "tensor", "kernel": "k_gemm_tc (all predictor GEMMs)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": (achieved / peak) if achieved else None,
                         "peak_source": peak_source,
                         "frac_of_measured_burst": (achieved / peaks.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"])
                                                    if achieved and pc.precision != "fp8" else None),
                         "frac_of_nominal_dense": (achieved / 2250.0
                                                   if achieved and pc.precision != "fp8" else None),
                         "sm_mhz_median": clocks.get("sm_mhz"),
                         "traffic": (sum(GEMM_DRAM_BYTES_PER_LAUNCH_FULL) / 4
                                     if args.workload == "full" and not args.candidates
                                     and gemm_source_sha() == GEMM_TRAFFIC_SOURCE_SHA else None),
                         "traffic_unit": "DRAM bytes per launch (mean of the four per-layer GEMMs)",
                         "traffic_source": f"ncu capture of the GEMM source hashed {GEMM_TRAFFIC_SOURCE_SHA or '(none)'}; "
                                           f"current source {gemm_source_sha()}",
                         "gemm_share_of_step": (gemm_ms / prof_steps) / step_ms if gemm_launches else None,
                         "gemm_tflop_per_step": step_flops / 1e12 if step_flops else None},
            "step_roofline": step_roofline(pc, H, N * R * B, step_flops / 1e12 if step_flops else None,
                                           step_ms, peaks),
            "e2e": {"value": rollouts / (e2e_ms * 1e-3), "unit": "candidate rollouts/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline and world == 1:
            v, info = cpu_baseline(wl, budget_s=args.cpu_budget)
            line["cpu_baseline"] = {"value": v, "unit": "candidate rollouts/s", "cores": info["cores"],
                                    "kind": "oracle", "sample": info["sample"]}
            if not args.no_cpu_full_configs:
                line["cpu_baseline"]["full_configs"] = cpu_full_configs()
        elif world > 1:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    planner.close()
    if world > 1:
        dist.destroy_process_group()


def run_sharded(args, wl):
    """Strong scaling of one planning step: the B problems' candidates of every round split
    across the ranks (cem_search_transformer_gb300.sharded), one NCCL all-gather of the
    energies per round. The step runs through the library's per-call entry points (no plan
    graph), so at one rank it also measures what the graph saves."""
    import torch
    import torch.distributed as dist
    from cem_search_transformer_gb300 import binding, build_lib, sharded

    rank, world, local = rank_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_lib.build()
    pc = wl.predictor
    B, N, K, R, H = wl.B, wl.N, wl.K, wl.rounds, wl.horizon
    planner = binding.Planner(pc, max_horizon=H, device=local,
                              max_chunk=-(-N * B // world))
    planner.load_weights(synthetic.make_weights(pc, seed=0))
    z0, goal, s0 = synthetic.make_problems(pc, B)
    mu0, sg0 = synthetic.make_gaussian(pc, B, H)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hz0, hgoal, hs0, hmu, hsg = pin(z0), pin(goal), pin(s0), pin(mu0), pin(sg0)
    hout = torch.zeros(B, pc.action_dim).pin_memory()
    gather = sharded.torch_all_gather() if world > 1 else (lambda buf: [buf])
    backend = sharded.CudaBackend(planner)

    def step(host_io: bool):
        if host_io:
            ins = [x.to(dev, non_blocking=True) for x in (hz0, hs0, hgoal, hmu, hsg)]
        else:
            ins = dev_in
        action, _ = sharded.plan_sharded(backend, *ins, B, H, N, K, R, wl.seed, world, rank, gather)
        if host_io:
            hout.copy_(action, non_blocking=True)
        return action

    dev_in = [x.to(dev) for x in (hz0, hs0, hgoal, hmu, hsg)]
    for _ in range(args.warmup):
        step(False)
    planner.sync_check()
    times = {}
    with ClockSampler(local, args.clocks_dir) as clk:
        for host_io in (False, True):
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                step(host_io)
                if host_io:
                    torch.cuda.current_stream(dev).synchronize()
            e1.record()
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            times[host_io] = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
    planner.sync_check()
    rollouts = N * R * B
    if rank == 0:
        launches = planner.kernel_count(B, H, N, K, R)
        line = {
            "metric": METRIC, "value": rollouts / (times[False] * 1e-3), "unit": "candidate rollouts/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": times[False],
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) embeddings)",
            "config": {"workload": workload_desc(wl),
                       "parallelism": f"candidates of every round split over {world} ranks, one "
                                      "all-gather of B x N fp32 energies per round",
                       "launch": "per-call entry points (no plan graph)",
                       "l2": "not flushed: working set exceeds the 129 MB L2"},
            "e2e": {"value": rollouts / (times[True] * 1e-3), "unit": "candidate rollouts/s",
                    "ms_per_step": times[True],
                    "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (hz0, hgoal, hs0, hmu, hsg)),
                    "d2h_bytes_per_step": hout.numel() * hout.element_size()},
            "gpu_launches": launches * args.steps,
            "gpu_launches_note": "the plan graph's kernel count for the whole problem; a rank's "
                                 "share of the predictor kernels is smaller, its per-round context "
                                 "projection adds two",
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    planner.close()
    if world > 1:
        dist.destroy_process_group()


def run_closed_loop(args, wl):
    import torch
    from cem_search_transformer_gb300 import binding, build_lib

    build_lib.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pc = wl.predictor
    B, N, K, R, H, T = wl.B, wl.N, wl.K, wl.rounds, wl.horizon, args.closed_loop
    planner = binding.Planner(pc, max_horizon=H)
    planner.load_weights(synthetic.make_weights(pc, seed=0))
    z0, goal, s0 = synthetic.make_problems(pc, B)
    mu0, sg0 = synthetic.make_gaussian(pc, B, H)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    dz0, dgoal, ds0, dmu, dsg = t(z0), t(goal), t(s0), t(mu0), t(sg0)
    acts = torch.zeros(T, B, pc.action_dim, device=dev)
    dist = torch.zeros(T, B, device=dev)
    d0 = torch.zeros(B, device=dev)
    stream = torch.cuda.current_stream(dev)
    binding.energy_l1_noalloc(dz0, dgoal, B, 1, pc.patch_tokens, pc.embed_dim, d0, stream=stream)
    run = lambda: planner.closed_loop(dz0, ds0, dgoal, dmu, dsg, B, H, N, K, R, T, args.warm,
                                      wl.seed, acts, dist, stream=stream)
    for _ in range(max(1, args.warmup)):
        run()
    planner.sync_check(stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0, args.clocks_dir) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            run()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    planner.sync_check(stream)
    ms_episode = ev0.elapsed_time(ev1) / args.steps
    line = {
        "metric": "closed-loop control-step latency (plan + world-model step)",
        "value": ms_episode / T, "unit": "ms per control step", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16"
        if pc.precision == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(wl), "control_steps": T, "rounds": R,
                   "warm_start": bool(args.warm)},
        "distance_start": float(d0.mean().item()),
        "distance_per_step": [float(x) for x in dist.mean(dim=1).tolist()],
        "first_action_norm": [float(x) for x in acts[:, 0].norm(dim=1).tolist()],
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    planner.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="full", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--candidates", type=int, default=0,
                    help="override N (and K = N/10) of the workload: small cases for ncu captures")
    ap.add_argument("--rounds", type=int, default=0, help="override the workload's CEM rounds")
    ap.add_argument("--closed-loop", type=int, default=0, metavar="T",
                    help="time a T-step receding-horizon episode instead of one plan step")
    ap.add_argument("--warm", action="store_true", help="warm-start each step (--closed-loop)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the plan's kernels directly on the stream instead of replaying "
                         "its CUDA graph (for the graph-vs-stream comparison)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time: the cpu_baseline sample, or all timed steps of "
                         "--impl reference together")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-full-configs", action="store_true",
                    help="skip timing whole tiny and small planning steps with the oracle")
    ap.add_argument("--shard", default="problems", choices=["problems", "candidates"],
                    help="under torchrun: each rank plans its own problems (default), or every "
                         "rank scores a slice of one problem's candidates with one all-gather of "
                         "the energies per round")
    ap.add_argument("--clocks-dir", default="",
                    help="directory for the raw nvidia-smi samples (default: the temp directory)")
    args = ap.parse_args()
    wl = synthetic.WORKLOADS[args.workload]
    if args.candidates:
        import dataclasses
        wl = dataclasses.replace(wl, N=args.candidates, K=max(1, args.candidates // 10))
    if args.rounds:
        import dataclasses
        wl = dataclasses.replace(wl, rounds=args.rounds)
    if args.closed_loop:
        run_closed_loop(args, wl)
    elif args.impl == "reference":
        run_reference(args, wl)
    elif args.shard == "candidates":
        run_sharded(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
